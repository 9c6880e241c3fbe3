"""AllReduce for callers that cannot allocate, checked against the communicator path.

Some callers cannot call cudaMalloc at the moment they need a collective: a
framework whose caching allocator owns all device memory, a serving loop that
cannot afford cudaMalloc's implicit device synchronisation, a deployment held
to a fixed memory budget.  dcc_allreduce_noalloc serves them from one fixed
device array inside the library.  Here it is called through the C ABI twice in
a row -- different element types, sizes and in/out-of-place, so that anything
the first call leaves in the shared array would show in the second -- and each
result is compared with dcc_allreduce (two-shot via scratch, the same
schedule) on the same inputs, bit for bit, the tolerance every parity test in
this suite uses.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _lib_and_binding():
    from driven_collective_communication_gb300 import build
    build.build()
    from driven_collective_communication_gb300 import dcc
    lib = ctypes.CDLL(dcc.LIB_PATH)
    f = lib.dcc_allreduce_noalloc
    f.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                  ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f, dcc


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


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


def test_noalloc_matches_communicator_path_two_calls_in_a_row():
    noalloc, dcc = _lib_and_binding()
    from driven_collective_communication_gb300 import workloads as W

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream
    calls = [
        # (workload recipe, count, in place, dcc dtype code)
        (W.c3(64), 64 * 8192, False, dcc.DCC_BF16),                  # 1 MiB per rank
        (W.with_count(W.C2, 700001), 700001, True, dcc.DCC_INT32),   # ragged, in place
    ]
    for i, (w, count, inplace, code) in enumerate(calls):
        xs = [x.cuda() for x in W.rank_inputs(w)]
        expect = _reference(dcc, xs, code)
        ys = xs if inplace else [torch.full_like(x, 7) for x in xs]
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = noalloc(w.n_ranks, _ptrs(xs), _ptrs(ys), count, code, stream)
        assert rc == dcc.DCC_OK, dcc.dcc_error_string(rc)
        torch.cuda.synchronize()
        if i > 0:  # the first call on a device may load the library's module there
            assert torch.cuda.mem_get_info()[0] == free_before
        for r in range(w.n_ranks):
            assert torch.equal(ys[r].view(torch.int16) if ys[r].element_size() == 2 else ys[r],
                               expect[r].view(torch.int16) if expect[r].element_size() == 2
                               else expect[r]), (i, r)


def test_noalloc_rejects_messages_beyond_its_array():
    noalloc, dcc = _lib_and_binding()
    torch.cuda.set_device(0)
    limit = dcc.DCC_NOALLOC_MAX_BYTES // 2  # bf16 elements that fit
    xs = [torch.zeros(limit + 8, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ys = [torch.empty_like(x) for x in xs]
    stream = torch.cuda.current_stream().cuda_stream
    assert noalloc(2, _ptrs(xs), _ptrs(ys), limit + 8, dcc.DCC_BF16, stream) == dcc.DCC_ERR_UNSUPPORTED
    assert noalloc(2, _ptrs(xs), _ptrs(ys), limit, dcc.DCC_BF16, stream) == dcc.DCC_OK
    assert noalloc(0, _ptrs(xs), _ptrs(ys), 16, dcc.DCC_BF16, stream) == dcc.DCC_ERR_INVALID_ARG
    torch.cuda.synchronize()
