"""PortChannels and the host proxy, on the GPU, through the C ABI.

MSCCL++ README, "PortChannel and MemoryChannel" and "Host-Side Communication
Proxy": one GPU thread pushes triggers, a host proxy thread runs the copies
(cudaMemcpyAsync on copy engines) and the signals; a custom proxy handles
user-defined triggers (the README's fst = 1, 2, 0xdeadbeef example).
"""
import numpy as np
import pytest
import torch

import oracle
from driven_collective_communication_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dcc():
    from driven_collective_communication_gb300 import build
    build.build()
    from driven_collective_communication_gb300 import dcc as mod
    torch.cuda.set_device(0)
    return mod


def test_port_put_signal_flush(dcc, proxy_streams):
    n = 4
    with dcc.Comm(n) as comm:
        ins = [torch.arange(8192, dtype=torch.int32, device="cuda") + 100000 * r for r in range(n)]
        outs = [torch.full((8192,), -1, dtype=torch.int32, device="cuda") for _ in range(n)]
        comm.register_all("input", ins)
        comm.register_all("output", outs)
        with pytest.raises(dcc.DccError) as e:  # no proxy yet
            dcc.dcc_port_put(comm.handle, 1, 3, 0, 0, 16)
        assert e.value.code == dcc.DCC_ERR_INVALID_ARG
        dcc.dcc_proxy_start(comm.handle)
        dcc.dcc_port_put(comm.handle, 1, 3, 1024, 512, 4096, signal=True, flush=True)
        dcc.dcc_port_put(comm.handle, 2, 0, 0, 0, 32768, signal=False, flush=True)
        assert comm.check() == dcc.DCC_OK
        got = outs[3].cpu().numpy()
        assert np.array_equal(got[256:1280], ins[1].cpu().numpy()[128:1152])
        assert np.all(got[:256] == -1) and np.all(got[1280:] == -1)
        assert np.array_equal(outs[0].cpu().numpy(), ins[2].cpu().numpy())
        assert dcc.dcc_proxy_stop(comm.handle) == dcc.DCC_OK
        rc, processed, custom = dcc.dcc_proxy_stats(comm.handle)
        assert rc == dcc.DCC_OK and processed == 4 and custom == 0  # 2 puts + 2 flushes


@pytest.fixture(params=[1, 4])
def proxy_streams(request, monkeypatch):
    """The proxy with one stream, and with copies spread over four (the default)."""
    monkeypatch.setenv("DCC_PROXY_STREAMS", str(request.param))
    return request.param


@pytest.mark.parametrize("n,m", [(8, 4096), (8, 4194304), (3, 1000 * 8), (16, 65536)])
def test_port_allgather_matches_oracle_and_memory_channel(dcc, proxy_streams, n, m):
    w = W.with_count(W.C5, n * m, n_ranks=n)
    xs = [x[:m].cuda() for x in W.rank_inputs(w)]
    port_out = [torch.full((n * m,), float("nan"), dtype=torch.float16, device="cuda") for _ in range(n)]
    mem_out = [torch.empty(n * m, dtype=torch.float16, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", xs)
        comm.register_all("output", port_out)   # first OUTPUT windows: the PortChannel targets
        comm.register_all("output", mem_out)
        dcc.dcc_proxy_start(comm.handle)
        for _ in range(3):  # repeated: semaphores and FIFO carry on without reset
            dcc.dcc_port_allgather(comm.handle, xs, port_out, m, "fp16")
        comm.allgather(xs, mem_out)
        rc = comm.check()
        if rc != dcc.DCC_OK:
            print("error detail", dcc.dcc_comm_error_detail(comm.handle))
            print(dcc.dcc_proxy_state(comm.handle, n))
        assert rc == dcc.DCC_OK
        assert dcc.dcc_proxy_stop(comm.handle) == dcc.DCC_OK
    expect = oracle.allgather([W.to_storage(x) for x in xs], "fp16")
    for r in range(n):
        assert np.array_equal(W.to_storage(port_out[r]), expect), r
        assert torch.equal(port_out[r].view(torch.int16), mem_out[r].view(torch.int16))


def test_fifo_wraps_around(dcc, proxy_streams):
    """Many more triggers than FIFO slots (1024): flow control on the tail."""
    n, m = 8, 2048
    xs = [torch.randn(m, device="cuda").half() for _ in range(n)]
    ys = [torch.empty(n * m, dtype=torch.float16, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        dcc.dcc_proxy_start(comm.handle)
        for _ in range(100):  # 100 x 8 ranks x (8 puts + 1 flush) = 7200 triggers
            dcc.dcc_port_allgather(comm.handle, xs, ys, m, "fp16")
        rc = comm.check()
        if rc != dcc.DCC_OK:
            print("error detail", dcc.dcc_comm_error_detail(comm.handle))
            st = dcc.dcc_proxy_state(comm.handle, n)
            print({k: st[k] for k in ("head", "tail", "done", "processed", "error")})
            print(st["signals"].tolist(), st["waits"].tolist())
        assert rc == dcc.DCC_OK
        assert dcc.dcc_proxy_stop(comm.handle) == dcc.DCC_OK
        rc, processed, _ = dcc.dcc_proxy_stats(comm.handle)
        assert processed == 7200
    ref = torch.cat(xs).view(torch.int16)
    for y in ys:
        assert torch.equal(y.view(torch.int16), ref)


def test_custom_proxy_handler(dcc):
    """The README's custom proxy: the GPU pushes 1, 2, 0xdeadbeef; the host
    handler receives them in order."""
    seen = []
    with dcc.Comm(2) as comm:
        dcc.dcc_proxy_set_handler(comm.handle, lambda fst, snd: seen.append((fst, snd)))
        dcc.dcc_proxy_start(comm.handle)
        dcc.dcc_fifo_push(comm.handle, [1, 2, 0xDEADBEEF], [10, 20, 30])
        torch.cuda.synchronize()
        assert comm.check() == dcc.DCC_OK
        assert dcc.dcc_proxy_stop(comm.handle) == dcc.DCC_OK
        assert seen == [(1, 10), (2, 20), (0xDEADBEEF, 30)]
        assert dcc.dcc_proxy_stats(comm.handle)[2] == 3
        with pytest.raises(dcc.DccError):  # built-in bit set: not a custom trigger
            dcc.dcc_fifo_push(comm.handle, [1 << 63])


def test_port_lost_signal_times_out(dcc):
    n, m = 4, 4096
    xs = [torch.randn(m, device="cuda").half() for _ in range(n)]
    ys = [torch.empty(n * m, dtype=torch.float16, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        dcc.dcc_set_wait_timeout_us(comm.handle, 50000)
        dcc.dcc_debug_skip_signal(comm.handle, 2)
        dcc.dcc_proxy_start(comm.handle)
        dcc.dcc_port_allgather(comm.handle, xs, ys, m, "fp16")
        assert comm.check() == dcc.DCC_ERR_TIMEOUT
        assert dcc.dcc_comm_error_detail(comm.handle)[1] == 2  # someone waited on rank 2
        assert dcc.dcc_proxy_stop(comm.handle) == dcc.DCC_OK
