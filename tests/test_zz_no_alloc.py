"""AllReduce for callers that cannot allocate, checked against the communicator
path and the oracle.

Some callers cannot call cudaMalloc at the moment they need a collective: a
framework whose caching allocator owns all device memory, a serving loop that
cannot afford cudaMalloc's implicit device synchronisation, a deployment held
to a fixed memory budget.  dcc_allreduce_noalloc serves them from one fixed
device array inside the library.  Here it is called through the C ABI several
times in a row -- different rank counts (1, 3, 8, 16), element types, sizes and
in/out-of-place, so that anything one call leaves in the shared array would
show in the next -- and each result is compared with dcc_allreduce (two-shot via
scratch, the same schedule) on the same inputs and with the oracle, bit for bit,
the tolerance every parity test in this suite uses.  dcc_noalloc_check must
report success after each call, and a wait made to run out (one rank's signals
dropped by a test knob, in a child process) must be reported, not lost.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib_and_binding():
    from driven_collective_communication_gb300 import build
    build.build()
    from driven_collective_communication_gb300 import dcc
    lib = ctypes.CDLL(dcc.LIB_PATH)
    f = lib.dcc_allreduce_noalloc
    f.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                  ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    chk = lib.dcc_noalloc_check
    chk.argtypes = [ctypes.c_void_p] + [ctypes.POINTER(ctypes.c_int)] * 3
    chk.restype = ctypes.c_int
    return f, chk, dcc


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _reference(dcc, xs, dtype_code):
    """The existing entry point: a communicator, registered buffers, two-shot via scratch."""
    n = len(xs)
    ys = [torch.empty_like(x) for x in xs]
    scr = [torch.empty_like(x) for x in xs]
    with dcc.Comm(n) as comm:
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        comm.register_all("scratch", scr)
        dcc.dcc_allreduce(comm.handle, xs, ys, xs[0].numel(), dtype_code, "two_shot_scratch")
        assert comm.check() == dcc.DCC_OK
    return ys


def test_noalloc_matches_communicator_path_and_oracle_calls_in_a_row():
    noalloc, check, dcc = _lib_and_binding()
    from driven_collective_communication_gb300 import workloads as W

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream
    calls = [
        # (workload recipe, in place, dcc dtype code)
        (W.c3(64), False, dcc.DCC_BF16),                                    # 8 x 1 MiB
        (W.with_count(W.C2, 700001), True, dcc.DCC_INT32),                  # ragged, in place
        (W.with_count(W.C1, 12345, n_ranks=1), False, dcc.DCC_FP32),        # one rank: a copy
        (W.with_count(W.C5, 16 * 8192 + 3, n_ranks=16), False, dcc.DCC_FP16),  # 16 ranks
        (W.with_count(W.C1, 99999, n_ranks=3), True, dcc.DCC_FP32),         # 3 ranks, in place
        (W.with_count(W.c3(1), (4 << 20) // 2), False, dcc.DCC_BF16),       # the largest message
    ]
    for i, (w, inplace, code) in enumerate(calls):
        host = W.rank_inputs(w)
        expect_oracle = oracle.allreduce([W.to_storage(x) for x in host], w.dtype)
        xs = [x.cuda() for x in host]
        expect = _reference(dcc, xs, code)
        ys = xs if inplace else [torch.full_like(x, 7) for x in xs]
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = noalloc(w.n_ranks, _ptrs(xs), _ptrs(ys), w.count, code, stream)
        assert rc == dcc.DCC_OK, dcc.dcc_error_string(rc)
        r, p, b = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_int(-1)
        assert check(stream, ctypes.byref(r), ctypes.byref(p), ctypes.byref(b)) == dcc.DCC_OK, i
        if i > 0:  # the first call on a device may load the library's module there
            assert torch.cuda.mem_get_info()[0] == free_before, i
        for q in range(w.n_ranks):
            assert torch.equal(_bits(ys[q]), _bits(expect[q])), (i, q)
            assert np.array_equal(W.to_storage(ys[q]), expect_oracle), (i, q)


def test_noalloc_rejects_messages_beyond_its_array():
    noalloc, _, dcc = _lib_and_binding()
    torch.cuda.set_device(0)
    limit = dcc.DCC_NOALLOC_MAX_BYTES // 2  # bf16 elements that fit
    xs = [torch.zeros(limit + 8, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ys = [torch.empty_like(x) for x in xs]
    stream = torch.cuda.current_stream().cuda_stream
    assert noalloc(2, _ptrs(xs), _ptrs(ys), limit + 8, dcc.DCC_BF16, stream) == dcc.DCC_ERR_UNSUPPORTED
    assert noalloc(2, _ptrs(xs), _ptrs(ys), limit, dcc.DCC_BF16, stream) == dcc.DCC_OK
    assert noalloc(0, _ptrs(xs), _ptrs(ys), 16, dcc.DCC_BF16, stream) == dcc.DCC_ERR_INVALID_ARG
    assert dcc.dcc_noalloc_check(stream)[0] == dcc.DCC_OK


_CHILD = r"""
import sys
sys.path.insert(0, %(root)r)
import torch
from driven_collective_communication_gb300 import dcc
torch.cuda.set_device(0)
xs = [torch.ones(65536, dtype=torch.float32, device="cuda") for _ in range(4)]
ys = [torch.empty_like(x) for x in xs]
dcc.dcc_allreduce_noalloc(4, xs, ys, 65536, "fp32")
code, rank, peer, block = dcc.dcc_noalloc_check()
assert code == dcc.DCC_ERR_TIMEOUT, code
assert peer == 1 and rank in (0, 2, 3) and block >= 0, (rank, peer, block)
assert dcc.dcc_noalloc_check()[0] == dcc.DCC_OK  # reported once, then cleared
print("timeout reported", rank, peer, block)
"""


def test_noalloc_reports_a_wait_that_ran_out():
    """Rank 1 sends no signals (test knob, read at the first call on the device),
    so the other ranks' waits run out after 50 ms; dcc_noalloc_check reports
    the first of them with its rank, peer and block, then clears the record.
    Runs in a child process so the knob touches no other test."""
    _lib_and_binding()  # builds the library if needed
    env = dict(os.environ, DCC_NOALLOC_SKIP_SIGNAL="1", DCC_WAIT_TIMEOUT_US="50000")
    r = subprocess.run([sys.executable, "-c", _CHILD % {"root": ROOT}], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "timeout reported" in r.stdout
