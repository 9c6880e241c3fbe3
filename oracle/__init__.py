"""CPU oracle for the collectives -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
it never loads the product library.

Arrays cross this boundary as numpy arrays of raw element storage:
``int32`` -> ``np.int32``, ``fp32`` -> ``np.float32``, ``fp16`` and ``bf16``
-> ``np.uint16`` bit patterns.  The arithmetic lives in ``oracle.c``; see its
header for the definition and the readings it takes.
"""
import ctypes
import os

import numpy as np

from .build import LIB, build_oracle

DTYPES = {"int32": 0, "fp32": 1, "fp16": 2, "bf16": 3}
STORAGE = {"int32": np.int32, "fp32": np.float32, "fp16": np.uint16, "bf16": np.uint16}

_lib = None


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB lets the mutation tests load a deliberately broken copy
        path = os.environ.get("ORACLE_LIB")
        if not path:
            build_oracle()
            path = LIB
        lib = ctypes.CDLL(path)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        lib.orc_allreduce.argtypes = [i32, ctypes.POINTER(vp), vp, sz, i32]
        lib.orc_allreduce_at.argtypes = [i32, ctypes.POINTER(vp), sz, i32, vp, sz, vp]
        lib.orc_allreduce_mt.argtypes = [i32, ctypes.POINTER(vp), vp, sz, i32, i32]
        lib.orc_reduce_scatter.argtypes = [i32, ctypes.POINTER(vp), vp, i32, sz, i32]
        lib.orc_allgather.argtypes = [i32, ctypes.POINTER(vp), vp, sz, i32]
        lib.orc_ring_barrier_counts.argtypes = [i32, ctypes.c_uint64, vp]
        lib.orc_convert_to_f32.argtypes = [vp, vp, sz, i32]
        lib.orc_convert_from_f32.argtypes = [vp, vp, sz, i32]
        lib.orc_linear_allreduce.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, sz, i32, vp]
        lib.orc_allreduce_op.argtypes = [i32, ctypes.POINTER(vp), vp, sz, i32, i32]
        lib.orc_linear_allreduce_residual.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                                      ctypes.POINTER(vp), sz, sz, i32, vp]
        lib.orc_linear_allreduce_tokens.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, sz, sz,
                                                    i32, vp]
        lib.orc_linear_allreduce_tokens_residual.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                                             ctypes.POINTER(vp), sz, sz, sz, i32, vp]
        for name in ("orc_allreduce", "orc_allreduce_at", "orc_allreduce_mt",
                     "orc_reduce_scatter", "orc_allgather", "orc_ring_barrier_counts",
                     "orc_convert_to_f32", "orc_convert_from_f32", "orc_linear_allreduce",
                     "orc_allreduce_op", "orc_linear_allreduce_residual", "orc_linear_allreduce_tokens",
                     "orc_linear_allreduce_tokens_residual"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _inputs(xs, dtype):
    if dtype not in DTYPES:
        raise ValueError("unknown dtype %r" % (dtype,))
    arrs = [np.ascontiguousarray(x, dtype=STORAGE[dtype]) for x in xs]
    if not arrs:
        raise ValueError("need at least one rank")
    n = len(arrs[0])
    if any(len(a) != n for a in arrs):
        raise ValueError("rank buffers differ in length")
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return arrs, ptrs, n


def _ok(rc, what):
    if rc != 0:
        raise ValueError("oracle %s rejected its arguments" % what)


def allreduce(xs, dtype, nthreads=1):
    """out[i] = R(sum over ranks in order 0..N-1 of xs[p][i]) (one output; all ranks equal)."""
    lib = _load()
    arrs, ptrs, n = _inputs(xs, dtype)
    out = np.empty(n, dtype=STORAGE[dtype])
    if nthreads > 1:
        rc = lib.orc_allreduce_mt(len(arrs), ptrs, out.ctypes.data, n, DTYPES[dtype], nthreads)
    else:
        rc = lib.orc_allreduce(len(arrs), ptrs, out.ctypes.data, n, DTYPES[dtype])
    _ok(rc, "allreduce")
    return out


OPS = {"max": 1, "min": 2}


def allreduce_op(xs, dtype, op):
    """out[i] = the IEEE maximum / minimum over ranks (in order 0..N-1) of xs[p][i];
    op is "max" or "min" (the sum is ``allreduce``)."""
    lib = _load()
    arrs, ptrs, n = _inputs(xs, dtype)
    out = np.empty(n, dtype=STORAGE[dtype])
    _ok(lib.orc_allreduce_op(len(arrs), ptrs, out.ctypes.data, n, DTYPES[dtype], OPS[op]), "allreduce_op")
    return out


def allreduce_at(xs, dtype, idx):
    """The AllReduce definition evaluated at the given element indices only."""
    lib = _load()
    arrs, ptrs, n = _inputs(xs, dtype)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(len(idx), dtype=STORAGE[dtype])
    _ok(lib.orc_allreduce_at(len(arrs), ptrs, n, DTYPES[dtype], idx.ctypes.data, len(idx),
                             out.ctypes.data), "allreduce_at")
    return out


def reduce_scatter(xs, dtype, rank, recv_count):
    """Rank ``rank``'s ReduceScatter output: R(sum_p xs[p][rank*m : (rank+1)*m])."""
    lib = _load()
    arrs, ptrs, n = _inputs(xs, dtype)
    if (rank + 1) * recv_count > n:
        raise ValueError("recv_count too large for the inputs")
    out = np.empty(recv_count, dtype=STORAGE[dtype])
    _ok(lib.orc_reduce_scatter(len(arrs), ptrs, out.ctypes.data, rank, recv_count,
                               DTYPES[dtype]), "reduce_scatter")
    return out


def allgather(xs, dtype):
    """Every rank's AllGather output: xs[0] | xs[1] | ... | xs[N-1]."""
    lib = _load()
    arrs, ptrs, n = _inputs(xs, dtype)
    out = np.empty(n * len(arrs), dtype=STORAGE[dtype])
    _ok(lib.orc_allgather(len(arrs), ptrs, out.ctypes.data, n, DTYPES[dtype]), "allgather")
    return out


def ring_barrier_counts(n, iters):
    """N x N matrix [dst, src] of signals rank dst has received from rank src."""
    lib = _load()
    out = np.empty((n, n), dtype=np.uint64)
    _ok(lib.orc_ring_barrier_counts(n, iters, out.ctypes.data), "ring_barrier_counts")
    return out


def to_f32(bits, dtype):
    """Widen raw fp16/bf16 bit patterns to float32 (exact)."""
    lib = _load()
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(len(bits), dtype=np.float32)
    _ok(lib.orc_convert_to_f32(bits.ctypes.data, out.ctypes.data, len(bits), DTYPES[dtype]),
        "to_f32")
    return out


def from_f32(vals, dtype):
    """Narrow float32 values to fp16/bf16 bit patterns, round to nearest even."""
    lib = _load()
    vals = np.ascontiguousarray(vals, dtype=np.float32)
    out = np.empty(len(vals), dtype=np.uint16)
    _ok(lib.orc_convert_from_f32(vals.ctypes.data, out.ctypes.data, len(vals), DTYPES[dtype]),
        "from_f32")
    return out


def linear_allreduce(ws, xs, dtype, rows, kp):
    """y[i] = R(sum_p sum_k W_p[i, k] x_p[k]) for rank weights ws[p] (rows*kp,
    row-major) and inputs xs[p] (kp): the row-parallel linear layer + AllReduce."""
    lib = _load()
    if dtype not in ("fp16", "bf16"):
        raise ValueError("fp16 or bf16 only")
    warrs = [np.ascontiguousarray(a, dtype=np.uint16) for a in ws]
    xarrs = [np.ascontiguousarray(a, dtype=np.uint16) for a in xs]
    if len(warrs) != len(xarrs) or any(len(a) != rows * kp for a in warrs) or any(len(a) != kp for a in xarrs):
        raise ValueError("shapes")
    wp = (ctypes.c_void_p * len(warrs))(*[a.ctypes.data for a in warrs])
    xp = (ctypes.c_void_p * len(xarrs))(*[a.ctypes.data for a in xarrs])
    out = np.empty(rows, dtype=np.uint16)
    _ok(lib.orc_linear_allreduce(len(warrs), wp, xp, rows, kp, DTYPES[dtype], out.ctypes.data),
        "linear_allreduce")
    return out


def linear_allreduce_residual(ws, xs, res, dtype, rows, kp):
    """y_q[i] = R(sum_p sum_k W_p[i, k] x_p[k] + res_q[i]) for every rank q: the
    row-parallel linear layer + AllReduce with a residual per output rank,
    added before the one rounding.  Returns the N outputs as a list."""
    lib = _load()
    if dtype not in ("fp16", "bf16"):
        raise ValueError("fp16 or bf16 only")
    warrs = [np.ascontiguousarray(a, dtype=np.uint16) for a in ws]
    xarrs = [np.ascontiguousarray(a, dtype=np.uint16) for a in xs]
    rarrs = [np.ascontiguousarray(a, dtype=np.uint16) for a in res]
    n = len(warrs)
    if (len(xarrs) != n or len(rarrs) != n or any(len(a) != rows * kp for a in warrs)
            or any(len(a) != kp for a in xarrs) or any(len(a) != rows for a in rarrs)):
        raise ValueError("shapes")
    wp = (ctypes.c_void_p * n)(*[a.ctypes.data for a in warrs])
    xp = (ctypes.c_void_p * n)(*[a.ctypes.data for a in xarrs])
    rp = (ctypes.c_void_p * n)(*[a.ctypes.data for a in rarrs])
    out = np.empty(n * rows, dtype=np.uint16)
    _ok(lib.orc_linear_allreduce_residual(n, wp, xp, rp, rows, kp, DTYPES[dtype], out.ctypes.data),
        "linear_allreduce_residual")
    return [out[q * rows:(q + 1) * rows].copy() for q in range(n)]


def linear_allreduce_tokens(ws, xs, dtype, tokens, rows, kp):
    """Y[t, i] = R(sum_p sum_k W_p[i, k] X_p[t, k]) for rank weights ws[p]
    (rows*kp, row-major) and inputs xs[p] (tokens*kp, row-major): the
    row-parallel linear layer + AllReduce over a batch of tokens.  Returns
    tokens*rows elements, row-major (token t's outputs contiguous)."""
    lib = _load()
    if dtype not in ("fp16", "bf16"):
        raise ValueError("fp16 or bf16 only")
    warrs = [np.ascontiguousarray(a, dtype=np.uint16).ravel() for a in ws]
    xarrs = [np.ascontiguousarray(a, dtype=np.uint16).ravel() for a in xs]
    if (len(warrs) != len(xarrs) or any(len(a) != rows * kp for a in warrs)
            or any(len(a) != tokens * kp for a in xarrs)):
        raise ValueError("shapes")
    wp = (ctypes.c_void_p * len(warrs))(*[a.ctypes.data for a in warrs])
    xp = (ctypes.c_void_p * len(xarrs))(*[a.ctypes.data for a in xarrs])
    out = np.empty(tokens * rows, dtype=np.uint16)
    _ok(lib.orc_linear_allreduce_tokens(len(warrs), wp, xp, tokens, rows, kp, DTYPES[dtype], out.ctypes.data),
        "linear_allreduce_tokens")
    return out


def linear_allreduce_tokens_residual(ws, xs, res, dtype, tokens, rows, kp):
    """Y_q[t, i] = R(sum_p sum_k W_p[i, k] X_p[t, k] + res_q[t, i]) for every
    rank q (res_q tokens*rows, row-major like the output), the residual added
    before the one rounding.  Returns the N outputs as a list."""
    lib = _load()
    if dtype not in ("fp16", "bf16"):
        raise ValueError("fp16 or bf16 only")
    warrs = [np.ascontiguousarray(a, dtype=np.uint16).ravel() for a in ws]
    xarrs = [np.ascontiguousarray(a, dtype=np.uint16).ravel() for a in xs]
    rarrs = [np.ascontiguousarray(a, dtype=np.uint16).ravel() for a in res]
    n = len(warrs)
    if (len(xarrs) != n or len(rarrs) != n or any(len(a) != rows * kp for a in warrs)
            or any(len(a) != tokens * kp for a in xarrs) or any(len(a) != tokens * rows for a in rarrs)):
        raise ValueError("shapes")
    wp = (ctypes.c_void_p * n)(*[a.ctypes.data for a in warrs])
    xp = (ctypes.c_void_p * n)(*[a.ctypes.data for a in xarrs])
    rp = (ctypes.c_void_p * n)(*[a.ctypes.data for a in rarrs])
    out = np.empty(n * tokens * rows, dtype=np.uint16)
    _ok(lib.orc_linear_allreduce_tokens_residual(n, wp, xp, rp, tokens, rows, kp, DTYPES[dtype], out.ctypes.data),
        "linear_allreduce_tokens_residual")
    return [out[q * tokens * rows:(q + 1) * tokens * rows].copy() for q in range(n)]


def library_path():
    return os.path.abspath(LIB)
