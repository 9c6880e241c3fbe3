"""Programmatic dependent launch keeps stream order: chains of dependent
collectives, each reading what the one before wrote, launched back to back
(no host synchronisation in between) with PDL on and off, eagerly and inside a
CUDA graph, give the oracle's bits at the end."""
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


N, M = 8, 4099            # ranks, ReduceScatter shard (ragged: 16,396-byte shards)
COUNT = N * M             # elements per rank of the AllReduces


def host(ts):
    return [t.cpu().numpy().copy() for t in ts]


def chain_expected(x0, rounds, ops):
    """The oracle applied step by step: AllReduce two-shot (x -> y), AllReduce
    one-shot (y -> x), ReduceScatter (x -> r), AllGather (r -> x), then MAX
    AllReduce (x -> y) and x = y + rank (a plain torch kernel in between)."""
    xs = [a.copy() for a in x0]
    for _ in range(rounds):
        y = oracle.allreduce(xs, "int32")
        xs = [y.copy() for _ in range(N)]
        x = oracle.allreduce(xs, "int32")
        xs = [x.copy() for _ in range(N)]
        rs = [oracle.reduce_scatter(xs, "int32", r, M) for r in range(N)]
        ag = oracle.allgather(rs, "int32")
        xs = [ag.copy() for _ in range(N)]
        if "max" in ops:
            y = oracle.allreduce_op(xs, "int32", "max")
            xs = [(y + np.int32(r)).astype(np.int32) for r in range(N)]
    return xs


def run_chain(dcc, comm, x, y, r, rounds, ops):
    h = comm.handle
    for _ in range(rounds):
        dcc.dcc_allreduce(h, x, y, COUNT, "int32", "two_shot")
        dcc.dcc_allreduce(h, y, x, COUNT, "int32", "one_shot")
        dcc.dcc_reduce_scatter(h, x, r, M, "int32")
        dcc.dcc_allgather(h, r, x, M, "int32")
        if "max" in ops:
            dcc.dcc_allreduce_op(h, x, y, COUNT, "int32", "max", "auto")
            for k in range(N):
                torch.add(y[k], k, out=x[k])


def make(dcc, seed):
    g = torch.Generator().manual_seed(seed)
    x0 = [torch.randint(-50, 51, (COUNT,), generator=g, dtype=torch.int32) for _ in range(N)]
    x = [t.cuda() for t in x0]
    y = [torch.empty_like(t) for t in x]
    r = [torch.empty(M, dtype=torch.int32, device="cuda") for _ in range(N)]
    comm = dcc.Comm(N)
    comm.register_all("input", x)
    comm.register_all("input", y)
    comm.register_all("input", r)
    comm.register_all("output", x)
    comm.register_all("output", y)
    comm.register_all("output", r)
    return comm, [a.numpy() for a in x0], x, y, r


@pytest.mark.parametrize("pdl", [True, False])
def test_eager_dependent_chain(dcc, pdl):
    rounds, ops = 6, ("max",)
    comm, x0, x, y, r = make(dcc, 31)
    try:
        dcc.dcc_set_pdl(comm.handle, pdl)
        run_chain(dcc, comm, x, y, r, rounds, ops)
        assert comm.check() == dcc.DCC_OK
        expect = chain_expected(x0, rounds, ops)
        got = host(x)
        for k in range(N):
            assert np.array_equal(got[k], expect[k]), k
    finally:
        comm.close()


def test_graph_dependent_chain(dcc):
    """The same chain captured into a CUDA graph with PDL on (the launches
    become programmatic edges) and replayed three times from fresh inputs."""
    rounds, ops = 2, ("max",)
    comm, x0, x, y, r = make(dcc, 32)
    try:
        dcc.dcc_set_pdl(comm.handle, True)
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            run_chain(dcc, comm, x, y, r, 1, ops)  # warm-up outside the capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            run_chain(dcc, comm, x, y, r, rounds, ops)
        expect = chain_expected(x0, rounds, ops)
        for _ in range(3):
            for k in range(N):
                x[k].copy_(torch.from_numpy(x0[k]))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            got = host(x)
            for k in range(N):
                assert np.array_equal(got[k], expect[k]), k
        assert comm.check() == dcc.DCC_OK
    finally:
        comm.close()


@pytest.mark.parametrize("kp,kernel", [(1024, "thread"), (1024, "tensor"), (4096, "bulk"), (4096, "tensor")])
def test_fused_layer_chain(dcc, monkeypatch, kp, kernel):
    """Fused linear layers feeding one another (rows == kp, y of one layer is x
    of the next) with PDL, on each kernel (thread loads, bulk copies, tensor
    cores: the last prefetches weights into L2 before its dependent-launch
    wait, and must read its input only after it).  Weights are permutations
    on rank 0 and zero elsewhere, so values neither grow nor round; the oracle
    follows the chain."""
    monkeypatch.setenv("DCC_FUSED_KERNEL", kernel)
    n, steps = 4, 8
    gen = np.random.default_rng(5)
    perms = [gen.permutation(kp) for _ in range(2)]

    def weights(perm):
        w0 = np.zeros((kp, kp), dtype=np.float32)
        w0[np.arange(kp), perm] = 1.0
        ws = [w0] + [np.zeros((kp, kp), dtype=np.float32) for _ in range(n - 1)]
        return [torch.from_numpy(w).to(torch.bfloat16) for w in ws]

    wsets = [weights(p) for p in perms]
    x0 = torch.from_numpy(gen.integers(-100, 101, size=kp).astype(np.float32)).to(torch.bfloat16)
    bufs = [[x0.clone().cuda() for _ in range(n)], [torch.empty(kp, dtype=torch.bfloat16, device="cuda")
                                                     for _ in range(n)]]
    wdev = [[w.cuda().reshape(-1) for w in ws] for ws in wsets]
    with dcc.Comm(n) as comm:
        for ws in wdev:
            comm.register_all("input", ws)
        comm.register_all("input", bufs[0])
        comm.register_all("input", bufs[1])
        comm.register_all("output", bufs[0])
        comm.register_all("output", bufs[1])
        dcc.dcc_set_pdl(comm.handle, True)
        for s in range(steps):
            src, dst = bufs[s % 2], bufs[(s + 1) % 2]
            dcc.dcc_linear_allreduce(comm.handle, wdev[s % 2], src, dst, kp, kp, "bf16")
        assert comm.check() == dcc.DCC_OK
        xs = [W.to_storage(x0) for _ in range(n)]
        for s in range(steps):
            ws = [W.to_storage(w.reshape(-1)) for w in wsets[s % 2]]
            y = oracle.linear_allreduce(ws, xs, "bf16", kp, kp)
            xs = [y.copy() for _ in range(n)]
        final = bufs[steps % 2]
        for k in range(n):
            assert np.array_equal(W.to_storage(final[k]), xs[k]), k
