"""Python binding of libdcc (include/dcc.h): argument marshalling only.

Every function here has the C name of the entry point it wraps and does
nothing but convert arguments (tensors -> device pointers, streams -> handles)
and raise ``DccError`` on a non-zero return.  All collective work runs in the
library's kernels.  Importing this module fails loudly when ``libdcc.so`` has
not been built -- there is no fallback path.

``Comm`` is a small convenience layer over the same calls for code that holds
torch tensors.
"""
import ctypes
import os

import torch  # loads the CUDA runtime that libdcc shares

_HERE = os.path.dirname(os.path.abspath(__file__))
# DCC_CHECK_BOUNDS=1 in the environment selects the bounds-checked build of the
# same library (every kernel data access checked; build with build(checked=True))
CHECKED = os.environ.get("DCC_CHECK_BOUNDS", "0") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "libdcc_checked.so" if CHECKED else "libdcc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("%s is not built (expected at %s); run "
                      "`python -c 'import __graft_entry__ as g; g.build()'` first"
                      % (os.path.basename(LIB_PATH), LIB_PATH))
_lib = ctypes.CDLL(LIB_PATH)

# ------------------------------------------------------------------ constants (dcc.h)
DCC_OK = 0
DCC_ERR_INVALID_ARG = -1
DCC_ERR_NOT_REGISTERED = -2
DCC_ERR_MISALIGNED = -3
DCC_ERR_NO_CHANNEL = -4
DCC_ERR_CUDA = -5
DCC_ERR_LAUNCH = -6
DCC_ERR_TIMEOUT = -7
DCC_ERR_UNSUPPORTED = -8
DCC_ERR_BOUNDS = -9

DCC_INT32, DCC_FP32, DCC_FP16, DCC_BF16 = 0, 1, 2, 3
DCC_ALGO_AUTO, DCC_ALGO_ONE_SHOT, DCC_ALGO_TWO_SHOT, DCC_ALGO_TWO_SHOT_SCRATCH = 0, 1, 2, 3
DCC_ALGO_TWO_SHOT_BULK = 4
DCC_ALGO_ONE_SHOT_LL = 5
DCC_LL_MAX_BYTES = 256 << 10
DCC_BUF_INPUT, DCC_BUF_OUTPUT, DCC_BUF_SCRATCH = 0, 1, 2
DCC_MAX_RANKS = 16
DCC_MAX_BLOCKS_PER_RANK = 128

DTYPE_CODES = {"int32": DCC_INT32, "fp32": DCC_FP32, "fp16": DCC_FP16, "bf16": DCC_BF16}
TORCH_CODES = {torch.int32: DCC_INT32, torch.float32: DCC_FP32, torch.float16: DCC_FP16,
               torch.bfloat16: DCC_BF16}
DCC_OP_SUM, DCC_OP_MAX, DCC_OP_MIN = 0, 1, 2
OP_CODES = {"sum": DCC_OP_SUM, "max": DCC_OP_MAX, "min": DCC_OP_MIN}
ALGO_CODES = {"auto": DCC_ALGO_AUTO, "one_shot": DCC_ALGO_ONE_SHOT, "two_shot": DCC_ALGO_TWO_SHOT,
              "two_shot_scratch": DCC_ALGO_TWO_SHOT_SCRATCH, "two_shot_bulk": DCC_ALGO_TWO_SHOT_BULK,
              "one_shot_ll": DCC_ALGO_ONE_SHOT_LL}
KIND_CODES = {"input": DCC_BUF_INPUT, "output": DCC_BUF_OUTPUT, "scratch": DCC_BUF_SCRATCH}

# ------------------------------------------------------------------ signatures
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_i = ctypes.c_int
_u64 = ctypes.c_uint64
_PP = ctypes.POINTER(ctypes.c_void_p)

_SIGS = {
    "dcc_comm_create": [_i, ctypes.POINTER(_vp)],
    "dcc_comm_destroy": [_vp],
    "dcc_register_buffer": [_vp, _i, _i, _vp, _sz],
    "dcc_memory_channel_make": [_vp, _i, _i],
    "dcc_allreduce": [_vp, _PP, _PP, _sz, _i, _i, _vp],
    "dcc_reduce_scatter": [_vp, _PP, _PP, _sz, _i, _vp],
    "dcc_allreduce_op": [_vp, _PP, _PP, _sz, _i, _i, _i, _vp],
    "dcc_reduce_scatter_op": [_vp, _PP, _PP, _sz, _i, _i, _vp],
    "dcc_allgather": [_vp, _PP, _PP, _sz, _i, _vp],
    "dcc_allreduce_from_host": [_vp, _PP, _PP, _PP, _PP, _sz, _i, _i, _vp],
    "dcc_ring_barrier": [_vp, _i, _vp],
    "dcc_comm_check": [_vp, _vp],
    "dcc_comm_error_detail": [_vp, ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i)],
    "dcc_channel_put": [_vp, _i, _i, _sz, _sz, _sz, _i, _vp],
    "dcc_channel_get": [_vp, _i, _i, _sz, _sz, _sz, _vp],
    "dcc_comm_read_semaphores": [_vp, _i, _vp, _vp, _vp],
    "dcc_set_wait_timeout_us": [_vp, _u64],
    "dcc_set_blocks_per_rank": [_vp, _i],
    "dcc_set_algo_threshold": [_vp, _i, _sz],
    "dcc_set_entry_barrier": [_vp, _i],
    "dcc_set_pdl": [_vp, _i],
    "dcc_select_algo": [_vp, _sz, _i, ctypes.POINTER(_i)],
    "dcc_auto_threshold": [_i, _i, ctypes.POINTER(_sz)],
    "dcc_debug_skip_signal": [_vp, _i],
    "dcc_launch_shape": [_vp, _sz, _i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)],
    "dcc_shard_range": [_sz, _i, _i, _sz, ctypes.POINTER(_sz), ctypes.POINTER(_sz)],
    "dcc_allreduce_noalloc": [_i, _PP, _PP, _sz, _i, _vp],
    "dcc_noalloc_check": [_vp, ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i)],
    "dcc_kernel_binary_version": [ctypes.POINTER(_i)],
    "dcc_proxy_start": [_vp],
    "dcc_proxy_stop": [_vp],
    "dcc_proxy_set_handler": [_vp, _vp, _vp],
    "dcc_proxy_stats": [_vp, _vp, _vp],
    "dcc_port_put": [_vp, _i, _i, _sz, _sz, _sz, _i, _i, _vp],
    "dcc_port_allgather": [_vp, _PP, _PP, _sz, _i, _vp],
    "dcc_fifo_push": [_vp, _vp, _vp, _i, _vp],
    "dcc_proxy_state": [_vp, _vp, _i],
    "dcc_linear_allreduce": [_vp, _PP, _PP, _PP, _sz, _sz, _i, _vp],
    "dcc_linear_allreduce_residual": [_vp, _PP, _PP, _PP, _PP, _sz, _sz, _i, _vp],
    "dcc_linear_allreduce_tokens": [_vp, _PP, _PP, _PP, _sz, _sz, _sz, _i, _vp],
    "dcc_linear_allreduce_tokens_residual": [_vp, _PP, _PP, _PP, _PP, _sz, _sz, _sz, _i, _vp],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _i
_lib.dcc_error_string.argtypes = [_i]
_lib.dcc_error_string.restype = ctypes.c_char_p
_lib.dcc_version.argtypes = []
_lib.dcc_version.restype = ctypes.c_char_p


class DccError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (what, dcc_error_string(code), code))


def _check(rc, what):
    if rc != DCC_OK:
        raise DccError(rc, what)
    return rc


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


def _ptrs(xs):
    return (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, torch.cuda.Stream):
        return s.cuda_stream
    return int(s)


def _code(table, v, what):
    if isinstance(v, int):
        return v
    if v in table:
        return table[v]
    raise ValueError("unknown %s %r" % (what, v))


def _dtype(v):
    if isinstance(v, torch.dtype):
        return TORCH_CODES[v]
    return _code(DTYPE_CODES, v, "dtype")


# ------------------------------------------------------------------ C entry points
def dcc_error_string(code):
    return _lib.dcc_error_string(int(code)).decode()


def dcc_version():
    return _lib.dcc_version().decode()


def dcc_comm_create(n_ranks):
    h = ctypes.c_void_p()
    _check(_lib.dcc_comm_create(int(n_ranks), ctypes.byref(h)), "dcc_comm_create")
    return h


def dcc_comm_destroy(comm):
    return _check(_lib.dcc_comm_destroy(comm), "dcc_comm_destroy")


def dcc_register_buffer(comm, rank, kind, buf, nbytes=None):
    if nbytes is None:
        nbytes = buf.numel() * buf.element_size()
    return _check(_lib.dcc_register_buffer(comm, rank, _code(KIND_CODES, kind, "kind"), _ptr(buf),
                                           nbytes), "dcc_register_buffer")


def dcc_memory_channel_make(comm, src_rank, dst_rank):
    return _check(_lib.dcc_memory_channel_make(comm, src_rank, dst_rank), "dcc_memory_channel_make")


def dcc_allreduce(comm, send, recv, count, dtype, algo="auto", stream=None):
    return _check(_lib.dcc_allreduce(comm, _ptrs(send), _ptrs(recv), count, _dtype(dtype),
                                     _code(ALGO_CODES, algo, "algo"), _stream(stream)),
                  "dcc_allreduce")


def dcc_reduce_scatter(comm, send, recv, recv_count, dtype, stream=None):
    return _check(_lib.dcc_reduce_scatter(comm, _ptrs(send), _ptrs(recv), recv_count, _dtype(dtype),
                                          _stream(stream)), "dcc_reduce_scatter")


def dcc_allreduce_op(comm, send, recv, count, dtype, op, algo="auto", stream=None):
    return _check(_lib.dcc_allreduce_op(comm, _ptrs(send), _ptrs(recv), count, _dtype(dtype),
                                        _code(OP_CODES, op, "op"), _code(ALGO_CODES, algo, "algo"),
                                        _stream(stream)), "dcc_allreduce_op")


def dcc_reduce_scatter_op(comm, send, recv, recv_count, dtype, op, stream=None):
    return _check(_lib.dcc_reduce_scatter_op(comm, _ptrs(send), _ptrs(recv), recv_count, _dtype(dtype),
                                             _code(OP_CODES, op, "op"), _stream(stream)),
                  "dcc_reduce_scatter_op")


def dcc_allgather(comm, send, recv, send_count, dtype, stream=None):
    return _check(_lib.dcc_allgather(comm, _ptrs(send), _ptrs(recv), send_count, _dtype(dtype),
                                     _stream(stream)), "dcc_allgather")


def dcc_allreduce_from_host(comm, host_send, host_recv, dev_send, dev_recv, count, dtype,
                            algo="auto", stream=None):
    return _check(_lib.dcc_allreduce_from_host(comm, _ptrs(host_send), _ptrs(host_recv),
                                               _ptrs(dev_send), _ptrs(dev_recv), count,
                                               _dtype(dtype), _code(ALGO_CODES, algo, "algo"),
                                               _stream(stream)), "dcc_allreduce_from_host")


def dcc_linear_allreduce(comm, weight, x, y, rows, kp, dtype, stream=None):
    return _check(_lib.dcc_linear_allreduce(comm, _ptrs(weight), _ptrs(x), _ptrs(y), rows, kp,
                                            _dtype(dtype), _stream(stream)), "dcc_linear_allreduce")


def dcc_linear_allreduce_residual(comm, weight, x, residual, y, rows, kp, dtype, stream=None):
    return _check(_lib.dcc_linear_allreduce_residual(comm, _ptrs(weight), _ptrs(x), _ptrs(residual), _ptrs(y),
                                                     rows, kp, _dtype(dtype), _stream(stream)),
                  "dcc_linear_allreduce_residual")


def dcc_linear_allreduce_tokens(comm, weight, x, y, tokens, rows, kp, dtype, stream=None):
    return _check(_lib.dcc_linear_allreduce_tokens(comm, _ptrs(weight), _ptrs(x), _ptrs(y), tokens, rows, kp,
                                                   _dtype(dtype), _stream(stream)),
                  "dcc_linear_allreduce_tokens")


def dcc_linear_allreduce_tokens_residual(comm, weight, x, residual, y, tokens, rows, kp, dtype, stream=None):
    return _check(_lib.dcc_linear_allreduce_tokens_residual(comm, _ptrs(weight), _ptrs(x), _ptrs(residual), _ptrs(y),
                                                            tokens, rows, kp, _dtype(dtype), _stream(stream)),
                  "dcc_linear_allreduce_tokens_residual")


def dcc_ring_barrier(comm, iters, stream=None):
    return _check(_lib.dcc_ring_barrier(comm, iters, _stream(stream)), "dcc_ring_barrier")


def dcc_comm_check(comm, stream=None):
    """Returns the status code (does not raise): DCC_OK or the device failure."""
    return _lib.dcc_comm_check(comm, _stream(stream))


def dcc_comm_error_detail(comm):
    r, p, b = _i(), _i(), _i()
    _check(_lib.dcc_comm_error_detail(comm, ctypes.byref(r), ctypes.byref(p), ctypes.byref(b)),
           "dcc_comm_error_detail")
    return r.value, p.value, b.value


def dcc_channel_put(comm, src, dst, remote_off, local_off, nbytes, signal=False, stream=None):
    return _check(_lib.dcc_channel_put(comm, src, dst, remote_off, local_off, nbytes,
                                       1 if signal else 0, _stream(stream)), "dcc_channel_put")


def dcc_channel_get(comm, src, dst, remote_off, local_off, nbytes, stream=None):
    return _check(_lib.dcc_channel_get(comm, src, dst, remote_off, local_off, nbytes,
                                       _stream(stream)), "dcc_channel_get")


def dcc_comm_read_semaphores(comm, n_ranks, block=0, stream=None):
    import numpy as np
    inbound = np.zeros((n_ranks, n_ranks), dtype=np.uint64)
    expected = np.zeros((n_ranks, n_ranks), dtype=np.uint64)
    _check(_lib.dcc_comm_read_semaphores(comm, block, inbound.ctypes.data, expected.ctypes.data,
                                         _stream(stream)), "dcc_comm_read_semaphores")
    return inbound, expected


def dcc_set_wait_timeout_us(comm, us):
    return _check(_lib.dcc_set_wait_timeout_us(comm, int(us)), "dcc_set_wait_timeout_us")


def dcc_set_blocks_per_rank(comm, blocks):
    return _check(_lib.dcc_set_blocks_per_rank(comm, int(blocks)), "dcc_set_blocks_per_rank")


def dcc_set_entry_barrier(comm, on):
    return _check(_lib.dcc_set_entry_barrier(comm, 1 if on else 0), "dcc_set_entry_barrier")


def dcc_set_pdl(comm, on):
    return _check(_lib.dcc_set_pdl(comm, 1 if on else 0), "dcc_set_pdl")


def dcc_set_algo_threshold(comm, dtype, nbytes):
    return _check(_lib.dcc_set_algo_threshold(comm, _dtype(dtype), int(nbytes)),
                  "dcc_set_algo_threshold")


def dcc_select_algo(comm, count, dtype):
    out = _i()
    _check(_lib.dcc_select_algo(comm, count, _dtype(dtype), ctypes.byref(out)), "dcc_select_algo")
    return {v: k for k, v in ALGO_CODES.items()}[out.value]


def dcc_auto_threshold(n_ranks, dtype):
    """Default one-shot threshold (bytes per rank) for n_ranks and dtype: the
    compiled crossover table (pure host logic)."""
    out = _sz()
    _check(_lib.dcc_auto_threshold(n_ranks, _dtype(dtype), ctypes.byref(out)), "dcc_auto_threshold")
    return out.value


def dcc_debug_skip_signal(comm, rank):
    return _check(_lib.dcc_debug_skip_signal(comm, int(rank)), "dcc_debug_skip_signal")


def dcc_launch_shape(comm, count, dtype, algo="auto"):
    b, t = _i(), _i()
    _check(_lib.dcc_launch_shape(comm, count, _dtype(dtype), _code(ALGO_CODES, algo, "algo"),
                                 ctypes.byref(b), ctypes.byref(t)), "dcc_launch_shape")
    return b.value, t.value


def dcc_shard_range(count, n_ranks, rank, elem_bytes):
    b, e = _sz(), _sz()
    _check(_lib.dcc_shard_range(count, n_ranks, rank, elem_bytes, ctypes.byref(b), ctypes.byref(e)),
           "dcc_shard_range")
    return b.value, e.value


def dcc_allreduce_noalloc(n_ranks, send, recv, count, dtype, stream=None):
    """AllReduce with no communicator and no allocation (see dcc.h)."""
    return _check(_lib.dcc_allreduce_noalloc(n_ranks, _ptrs(send), _ptrs(recv), count,
                                             _dtype(dtype), _stream(stream)),
                  "dcc_allreduce_noalloc")


def dcc_noalloc_check(stream=None):
    """Status of the allocation-free AllReduce on the current device: returns
    (code, rank, peer, block); code is DCC_OK or DCC_ERR_TIMEOUT (see dcc.h)."""
    r, p, b = _i(-1), _i(-1), _i(-1)
    rc = _lib.dcc_noalloc_check(_stream(stream), ctypes.byref(r), ctypes.byref(p), ctypes.byref(b))
    if rc not in (DCC_OK, DCC_ERR_TIMEOUT):
        raise DccError(rc, "dcc_noalloc_check")
    return rc, r.value, p.value, b.value


DCC_NOALLOC_MAX_BYTES = 4 << 20


def dcc_kernel_binary_version():
    """binaryVersion of the library's kernels on the current device (103 = sm_103a)."""
    v = _i()
    _check(_lib.dcc_kernel_binary_version(ctypes.byref(v)), "dcc_kernel_binary_version")
    return v.value

TRIGGER_HANDLER = ctypes.CFUNCTYPE(None, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p)
_handlers = {}  # keeps the ctypes callbacks alive per communicator


def dcc_proxy_start(comm):
    return _check(_lib.dcc_proxy_start(comm), "dcc_proxy_start")


def dcc_proxy_stop(comm):
    """Stops the proxy; returns its first error code (0 if none), does not raise."""
    return _lib.dcc_proxy_stop(comm)


def dcc_proxy_set_handler(comm, fn):
    """fn(fst, snd) runs on the proxy thread for every custom trigger (None removes it)."""
    key = comm.value if isinstance(comm, ctypes.c_void_p) else int(comm)
    cb = TRIGGER_HANDLER(lambda fst, snd, user: fn(fst, snd)) if fn is not None else None
    _handlers[key] = cb
    return _check(_lib.dcc_proxy_set_handler(comm, ctypes.cast(cb, ctypes.c_void_p) if cb else None,
                                             None), "dcc_proxy_set_handler")


def dcc_proxy_stats(comm):
    p, cu = ctypes.c_uint64(), ctypes.c_uint64()
    rc = _lib.dcc_proxy_stats(comm, ctypes.byref(p), ctypes.byref(cu))
    return rc, p.value, cu.value


def dcc_proxy_state(comm, n_ranks):
    """Diagnostic snapshot: dict with FIFO head/tail, flush word, counts and the
    port signal / wait matrices [dst][src]."""
    import numpy as np
    nw = 6 + 2 * n_ranks * n_ranks
    w = np.zeros(nw, dtype=np.uint64)
    _check(_lib.dcc_proxy_state(comm, w.ctypes.data, nw), "dcc_proxy_state")
    nn = n_ranks * n_ranks
    return {"head": int(w[0]), "tail": int(w[1]), "done": int(w[2]), "processed": int(w[3]),
            "custom": int(w[4]), "error": int(w[5].astype(np.int64)),
            "signals": w[6:6 + nn].reshape(n_ranks, n_ranks), "waits": w[6 + nn:].reshape(n_ranks, n_ranks)}


def dcc_port_put(comm, src, dst, remote_off, local_off, nbytes, signal=False, flush=False, stream=None):
    return _check(_lib.dcc_port_put(comm, src, dst, remote_off, local_off, nbytes, 1 if signal else 0,
                                    1 if flush else 0, _stream(stream)), "dcc_port_put")


def dcc_port_allgather(comm, send, recv, send_count, dtype, stream=None):
    return _check(_lib.dcc_port_allgather(comm, _ptrs(send), _ptrs(recv), send_count, _dtype(dtype),
                                          _stream(stream)), "dcc_port_allgather")


def dcc_fifo_push(comm, fst, snd=None, stream=None):
    n = len(fst)
    f = (ctypes.c_uint64 * n)(*fst)
    s = (ctypes.c_uint64 * n)(*snd) if snd is not None else None
    return _check(_lib.dcc_fifo_push(comm, f, s, n, _stream(stream)), "dcc_fifo_push")


def prepare_allreduce(comm, send, recv, count, dtype, algo="auto", stream=None):
    """Marshal the arguments of one dcc_allreduce once and return a callable that
    repeats exactly that call (for launch loops where Python overhead matters)."""
    args = (comm, _ptrs(send), _ptrs(recv), count, _dtype(dtype), _code(ALGO_CODES, algo, "algo"),
            _stream(stream))
    f = _lib.dcc_allreduce

    def call():
        rc = f(*args)
        if rc != DCC_OK:
            raise DccError(rc, "dcc_allreduce")
    return call


def prepare_linear_allreduce_tokens(comm, weight, x, y, tokens, rows, kp, dtype, stream=None):
    """Marshal the arguments of one dcc_linear_allreduce_tokens once and return
    a callable that repeats exactly that call."""
    args = (comm, _ptrs(weight), _ptrs(x), _ptrs(y), tokens, rows, kp, _dtype(dtype), _stream(stream))
    f = _lib.dcc_linear_allreduce_tokens

    def call():
        rc = f(*args)
        if rc != DCC_OK:
            raise DccError(rc, "dcc_linear_allreduce_tokens")
    return call


def raw_call(name, *args):
    """Call an entry point with raw ctypes arguments and return its code (tests of error paths)."""
    return getattr(_lib, name)(*args)


# ------------------------------------------------------------------ convenience
class Comm:
    """N virtual ranks on the current CUDA device, with all-pairs channels."""

    def __init__(self, n_ranks, connect="all"):
        self.n = n_ranks
        self.handle = dcc_comm_create(n_ranks)
        if connect == "all":
            for s in range(n_ranks):
                for d in range(n_ranks):
                    if s != d:
                        dcc_memory_channel_make(self.handle, s, d)
        elif connect == "ring":
            for s in range(n_ranks):
                if n_ranks > 1:
                    dcc_memory_channel_make(self.handle, s, (s + 1) % n_ranks)

    def register(self, rank, kind, tensor):
        dcc_register_buffer(self.handle, rank, kind, tensor)

    def register_all(self, kind, tensors):
        for r, t in enumerate(tensors):
            self.register(r, kind, t)

    def allreduce(self, send, recv=None, algo="auto", stream=None):
        recv = send if recv is None else recv
        dcc_allreduce(self.handle, send, recv, send[0].numel(), send[0].dtype, algo, stream)

    def reduce_scatter(self, send, recv, stream=None):
        dcc_reduce_scatter(self.handle, send, recv, recv[0].numel(), send[0].dtype, stream)

    def allreduce_op(self, send, recv=None, op="sum", algo="auto", stream=None):
        recv = send if recv is None else recv
        dcc_allreduce_op(self.handle, send, recv, send[0].numel(), send[0].dtype, op, algo, stream)

    def reduce_scatter_op(self, send, recv, op="sum", stream=None):
        dcc_reduce_scatter_op(self.handle, send, recv, recv[0].numel(), send[0].dtype, op, stream)

    def allgather(self, send, recv, stream=None):
        dcc_allgather(self.handle, send, recv, send[0].numel(), send[0].dtype, stream)

    def ring_barrier(self, iters, stream=None):
        dcc_ring_barrier(self.handle, iters, stream)

    def check(self, stream=None):
        return dcc_comm_check(self.handle, stream)

    def close(self):
        if self.handle is not None:
            dcc_comm_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
