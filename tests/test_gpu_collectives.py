"""GPU parity of the collectives against the CPU oracle, through the C ABI.

Every floating-point result is compared bit for bit: the kernels keep the
oracle's rank order and fp32 accumulation, so any correct schedule returns
the same bits (the tolerance of the method -- 1e-6*N*max|x| for fp32, 1 ulp of
the output type for fp16/bf16 -- is only needed for other orders and is never
used here).  int32 is exact by definition.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from driven_collective_communication_gb300 import workloads as W

pytestmark = pytest.mark.gpu

RECIPES = {"fp32": W.C1, "int32": W.C2, "bf16": W.C4, "fp16": W.C5}
ALGOS = ("one_shot", "two_shot", "two_shot_scratch", "two_shot_bulk", "one_shot_ll")


@pytest.fixture(scope="module")
def dcc():
    from driven_collective_communication_gb300 import build
    build.build()
    from driven_collective_communication_gb300 import dcc as mod
    torch.cuda.set_device(0)
    return mod


def same(got, expect, dtype):
    """Bit equality; NaN payloads may differ (only NaN-ness is compared)."""
    got = np.asarray(got)
    expect = np.asarray(expect)
    if dtype == "int32":
        return np.array_equal(got, expect)
    wide_g = oracle.to_f32(got, dtype) if dtype != "fp32" else got
    wide_e = oracle.to_f32(expect, dtype) if dtype != "fp32" else expect
    ng, ne = np.isnan(wide_g), np.isnan(wide_e)
    if not np.array_equal(ng, ne):
        return False
    return np.array_equal(got[~ng].view(np.uint32 if dtype == "fp32" else np.uint16),
                          expect[~ne].view(np.uint32 if dtype == "fp32" else np.uint16))


class Arena:
    """Per-rank input/output/scratch buffers registered once; cases use slices."""

    def __init__(self, dcc, n, elems_per_rank, elem_bytes=4):
        self.dcc = dcc
        self.n = n
        self.comm = dcc.Comm(n)
        nbytes = elems_per_rank * elem_bytes + 4096
        self.inp = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(n)]
        self.out = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(n)]
        self.scr = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(n)]
        for r in range(n):
            self.comm.register(r, "input", self.inp[r])
            self.comm.register(r, "output", self.out[r])
            self.comm.register(r, "scratch", self.scr[r])

    def view(self, bufs, dtype, count, offset=0):
        tdt = W.TORCH_DTYPES[dtype]
        eb = W.ELEM_BYTES[dtype]
        return [b[offset: offset + count * eb].view(tdt) for b in bufs]

    def close(self):
        self.comm.close()


def run_allreduce(dcc, arena, xs_host, dtype, algo, inplace, offset=0):
    """One AllReduce through the C ABI; None when the algorithm rejects the size
    (LL beyond its maximum, checked to be DCC_ERR_UNSUPPORTED)."""
    count = xs_host[0].numel()
    if algo == "one_shot_ll" and count * W.ELEM_BYTES[dtype] > dcc.DCC_LL_MAX_BYTES:
        send = arena.view(arena.inp, dtype, count, offset)
        with pytest.raises(dcc.DccError) as e:
            dcc.dcc_allreduce(arena.comm.handle, send, send, count, dtype, algo)
        assert e.value.code == dcc.DCC_ERR_UNSUPPORTED
        return None
    send = arena.view(arena.inp, dtype, count, offset)
    for r in range(arena.n):
        send[r].copy_(xs_host[r])
    recv = send if inplace else arena.view(arena.out, dtype, count, offset)
    if not inplace:
        for r in range(arena.n):
            recv[r].fill_(0)
    dcc.dcc_allreduce(arena.comm.handle, send, recv, count, dtype, algo)
    rc = arena.comm.check()
    assert rc == dcc.DCC_OK, dcc.dcc_error_string(rc)
    return [W.to_storage(t) for t in recv]


# ---------------------------------------------------------------- small parity sweep
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 16])
def test_allreduce_parity_sweep(dcc, n):
    """All dtypes x algorithms x in/out-of-place x counts (1 element, below one
    vector, ragged, several CTAs' worth + tail) against the oracle."""
    counts = [1, 5, 8, 16 * n + 3, 3 * 512 * 8 + 5, 70001]
    arena = Arena(dcc, n, max(counts))
    try:
        for dtype, recipe in RECIPES.items():
            for count in counts:
                w = W.with_count(recipe, count, n_ranks=n)
                xs = W.rank_inputs(w)
                expect = oracle.allreduce([W.to_storage(x) for x in xs], dtype)
                for algo in ALGOS:
                    for inplace in (False, True):
                        outs = run_allreduce(dcc, arena, xs, dtype, algo, inplace)
                        for r in range(n if outs is not None else 0):
                            assert same(outs[r], expect, dtype), (dtype, count, algo, inplace, r)
    finally:
        arena.close()


def test_empty_inputs_are_no_ops(dcc):
    """count 0: every entry point returns OK, launches nothing and leaves the
    outputs as they were."""
    n = 4
    xs = [torch.full((64,), float(r + 1), device="cuda") for r in range(n)]
    ys = [torch.full((64 * n,), -7.0, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        h = comm.handle
        for algo in ("auto", "one_shot", "two_shot", "two_shot_bulk", "one_shot_ll"):
            dcc.dcc_allreduce(h, xs, ys, 0, "fp32", algo)
        dcc.dcc_reduce_scatter(h, xs, ys, 0, "fp32")
        dcc.dcc_allgather(h, xs, ys, 0, "fp32")
        dcc.dcc_linear_allreduce(h, xs, xs, ys, 0, 8, "bf16")
        assert comm.check() == dcc.DCC_OK
    for y in ys:
        assert torch.all(y == -7.0)
    for r in range(n):
        assert torch.all(xs[r] == r + 1)


def test_random_configurations_match_oracle(dcc, monkeypatch):
    """Two hundred seeded random mixes of rank count (compiled and runtime-N instances),
    element count, dtype, algorithm, in/out of place, CTAs per rank, threads
    per CTA, the entry barrier and programmatic dependent launch, each against
    the oracle bit for bit."""
    rng = np.random.default_rng(2026)
    checked = 0
    for case in range(200):
        n = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16]))
        dtype = str(rng.choice(sorted(RECIPES)))
        count = int(rng.integers(1, 60000))
        algo = str(rng.choice(ALGOS))
        inplace = bool(rng.integers(0, 2))
        blocks = int(rng.choice([0, 1, 3, 17, 128]))
        threads = int(rng.choice([0, 64, 96, 256]))
        entry_barrier = bool(rng.integers(0, 4) == 0)
        pdl = bool(rng.integers(0, 2))
        if threads:
            monkeypatch.setenv("DCC_THREADS", str(threads))
        else:
            monkeypatch.delenv("DCC_THREADS", raising=False)
        w = W.with_count(RECIPES[dtype], count, n_ranks=n)
        xs = W.rank_inputs(w)
        expect = oracle.allreduce([W.to_storage(x) for x in xs], dtype)
        arena = Arena(dcc, n, count)
        try:
            h = arena.comm.handle
            dcc.dcc_set_blocks_per_rank(h, blocks)
            dcc.dcc_set_entry_barrier(h, entry_barrier)
            dcc.dcc_set_pdl(h, pdl)
            what = (case, n, dtype, count, algo, inplace, blocks, threads, entry_barrier, pdl)
            if entry_barrier and algo in ("two_shot_bulk", "one_shot_ll"):
                send = arena.view(arena.inp, dtype, count)
                with pytest.raises(dcc.DccError) as e:
                    dcc.dcc_allreduce(h, send, send, count, dtype, algo)
                assert e.value.code == dcc.DCC_ERR_UNSUPPORTED, what
                continue
            outs = run_allreduce(dcc, arena, xs, dtype, algo, inplace)
            for r in range(n if outs is not None else 0):
                assert same(outs[r], expect, dtype), (what, r)
            checked += outs is not None
        finally:
            arena.close()
    assert checked >= 150, checked  # most draws run (the rest are the rejected combinations)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_allreduce_special_values(dcc, dtype):
    """Raw random bit patterns: subnormals (no flush to zero), signed zeros,
    infinities, NaNs, overflow of the fp32 sum."""
    n, count = 8, 4099
    rng = np.random.default_rng(17)
    if dtype == "fp32":
        xs = [torch.from_numpy(rng.integers(0, 2 ** 32, size=count, dtype=np.uint64)
                               .astype(np.uint32).view(np.float32)) for _ in range(n)]
    else:
        xs = [W.from_storage(rng.integers(0, 2 ** 16, size=count, dtype=np.uint64).astype(np.uint16),
                             dtype) for _ in range(n)]
    # add a block of pure subnormals and -0.0 columns
    for r in range(n):
        if dtype == "fp32":
            xs[r][:64] = torch.tensor(np.full(64, 1e-45 * (r + 1), np.float32))
            xs[r][64:128] = -0.0
        else:
            sub = np.arange(1, 65, dtype=np.uint16) + r
            xs[r][:64] = W.from_storage(sub, dtype)
            xs[r][64:128] = W.from_storage(np.full(64, 0x8000, np.uint16), dtype)
    expect = oracle.allreduce([W.to_storage(x) for x in xs], dtype)
    arena = Arena(dcc, n, count)
    try:
        for algo in ALGOS:
            for inplace in (False, True):
                outs = run_allreduce(dcc, arena, xs, dtype, algo, inplace)
                for r in range(n if outs is not None else 0):
                    assert same(outs[r], expect, dtype), (algo, inplace, r)
    finally:
        arena.close()


def test_allgather_bulk_and_thread_paths_agree(dcc, monkeypatch):
    """The bulk-copy AllGather and the thread-copy AllGather produce the same bytes."""
    n, m = 8, 3 * 16384 // 2 + 8  # fp16: 48 KiB + 16 B per rank, several 16 KiB tiles + a partial one
    m = 2 * m  # > 64 KiB per rank: the bulk path
    xs = [torch.randn(m, device="cuda").half() for _ in range(n)]
    outs = {}
    for flag in ("1", "0"):
        monkeypatch.setenv("DCC_AG_BULK", flag)
        ys = [torch.full((n * m,), float("nan"), device="cuda").half() for _ in range(n)]
        with dcc.Comm(n) as comm:
            comm.register_all("input", xs)
            comm.register_all("output", ys)
            comm.allgather(xs, ys)
            assert comm.check() == dcc.DCC_OK
        outs[flag] = ys
    ref = torch.cat(xs).view(torch.int16)
    for r in range(n):
        assert torch.equal(outs["1"][r].view(torch.int16), ref)
        assert torch.equal(outs["0"][r].view(torch.int16), ref)


@pytest.mark.parametrize("n", [6, 8])
def test_allgather_launch_shapes(dcc, n):
    """The AllGather's vector path (several vectors in flight per thread) covers
    every element for any number of CTAs per rank, including a partial chunk."""
    m = 8 * (4096 * 8 * 3 + 517)  # bf16: 3 full 8-vector x 512-thread chunks + a ragged one
    xs = [torch.randn(m, device="cuda").to(torch.bfloat16) for _ in range(n)]
    ref = torch.cat(xs).view(torch.int16)
    ys = [torch.empty(n * m, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        for blocks in (1, 2, 7, 128, 0):
            dcc.dcc_set_blocks_per_rank(comm.handle, blocks)
            for y in ys:
                y.fill_(float("nan"))
            comm.allgather(xs, ys)
            assert comm.check() == dcc.DCC_OK
            for r in range(n):
                assert torch.equal(ys[r].view(torch.int16), ref), (blocks, r)


def test_launch_shape_does_not_change_bits(dcc):
    """Any number of CTAs per rank returns the same bits (fixed per-element order)."""
    n, count = 8, 123457
    w = W.with_count(W.C4, count)
    xs = W.rank_inputs(w)
    expect = oracle.allreduce([W.to_storage(x) for x in xs], "bf16")
    arena = Arena(dcc, n, count)
    try:
        for blocks in (1, 2, 7, 19, 128):
            dcc.dcc_set_blocks_per_rank(arena.comm.handle, blocks)
            for algo in ALGOS:
                for inplace in (False, True):
                    outs = run_allreduce(dcc, arena, xs, "bf16", algo, inplace)
                    assert outs is None or all(same(o, expect, "bf16") for o in outs), \
                        (blocks, algo, inplace)
    finally:
        arena.close()


# ---------------------------------------------------------------- the five workloads
def test_c1_fp32_n2_one_shot_full(dcc):
    w = W.C1
    xs = W.rank_inputs(w)
    expect = oracle.allreduce([W.to_storage(x) for x in xs], "fp32")
    exact = sum(W.to_storage(x).astype(np.int64) for x in xs)
    assert np.array_equal(expect.astype(np.int64), exact)
    arena = Arena(dcc, 2, w.count)
    try:
        outs = run_allreduce(dcc, arena, xs, "fp32", "one_shot", inplace=False)
        for o in outs:
            assert same(o, expect, "fp32")
    finally:
        arena.close()


def test_c2_int32_n8_inplace_both_algorithms_full(dcc):
    w = W.C2
    xs = [x for x in W.rank_inputs(w, device="cuda")]
    host = [W.to_storage(x) for x in xs]
    expect = oracle.allreduce(host, "int32", nthreads=16)
    comm = dcc.Comm(8)
    try:
        for algo in ("one_shot", "two_shot"):
            bufs = [x.clone() for x in xs]
            comm.register_all("input", bufs)
            comm.allreduce(bufs, bufs, algo=algo)
            assert comm.check() == dcc.DCC_OK
            for b in bufs:
                assert np.array_equal(W.to_storage(b), expect), algo
            del bufs
    finally:
        comm.close()


@pytest.mark.parametrize("tokens", W.C3_TOKENS)
def test_c3_bf16_decode_sizes(dcc, tokens):
    w = W.c3(tokens)
    xs = W.rank_inputs(w)
    expect = oracle.allreduce([W.to_storage(x) for x in xs], "bf16")
    arena = Arena(dcc, 8, w.count, elem_bytes=2)
    try:
        for algo in ALGOS:
            for inplace in (False, True):
                outs = run_allreduce(dcc, arena, xs, "bf16", algo, inplace=inplace)
                for o in outs or []:
                    assert same(o, expect, "bf16"), (algo, inplace)
    finally:
        arena.close()


def host_bits(t):
    """A device tensor's raw storage on the host, as unsigned integers (a view,
    no conversion), for whole-buffer bit comparisons."""
    a = W.to_storage(t)
    return a.view(np.uint16) if a.itemsize == 2 else a.view(np.uint32)


def test_c4_bf16_n8_256MiB_full(dcc):
    """Full size, the launch configuration the benchmark times (AUTO) and every
    other large-message schedule: all 8 x 134,217,728 outputs of every rank
    compared bit for bit with the oracle (threaded over the host cores), and
    every rank's output identical on the device."""
    w = W.C4
    xs = W.rank_inputs(w, device="cuda")
    recv = [torch.empty_like(x) for x in xs]
    comm = dcc.Comm(8)
    expect = oracle.allreduce([W.to_storage(x) for x in xs], "bf16", nthreads=os.cpu_count() or 1)
    expect = expect.view(np.uint16)
    try:
        comm.register_all("input", xs)
        comm.register_all("output", recv)
        for algo in ("auto", "two_shot", "two_shot_bulk"):
            for r in range(8):
                recv[r].fill_(0)
            comm.allreduce(xs, recv, algo=algo)
            assert comm.check() == dcc.DCC_OK
            for r in range(1, 8):
                assert torch.equal(recv[r].view(torch.int16), recv[0].view(torch.int16)), algo
            for r in range(8):
                got = host_bits(recv[r])
                assert np.array_equal(got, expect), (algo, r, int(np.count_nonzero(got != expect)))
    finally:
        comm.close()


@pytest.mark.parametrize("n,dtype", [(2, "bf16"), (4, "bf16"), (16, "bf16"), (8, "fp32")])
def test_256MiB_per_rank_other_rank_counts_and_fp32_full(dcc, n, dtype):
    """The other full-size AllReduces the benchmark times (256 MiB per rank, AUTO):
    every element of every rank's output against the oracle, bit for bit."""
    recipe = W.C4 if dtype == "bf16" else W.C1
    count = (256 << 20) // W.ELEM_BYTES[dtype]
    w = W.with_count(recipe, count, n_ranks=n)
    xs = W.rank_inputs(w, device="cuda")
    recv = [torch.empty_like(x) for x in xs]
    expect = oracle.allreduce([W.to_storage(x) for x in xs], dtype, nthreads=os.cpu_count() or 1)
    expect = expect.view(np.uint16 if dtype == "bf16" else np.uint32)
    bits = torch.int16 if dtype == "bf16" else torch.int32
    with dcc.Comm(n) as comm:
        comm.register_all("input", xs)
        comm.register_all("output", recv)
        comm.allreduce(xs, recv, algo="auto")
        assert comm.check() == dcc.DCC_OK
    for r in range(1, n):
        assert torch.equal(recv[r].view(bits), recv[0].view(bits)), r
    for r in range(n):
        got = host_bits(recv[r])
        assert np.array_equal(got, expect), (r, int(np.count_nonzero(got != expect)))


def test_c5_fp16_reduce_scatter_and_allgather_full(dcc):
    w = W.C5
    n = 8
    xs = W.rank_inputs(w, device="cuda")
    m = w.count // n
    rs_out = [torch.empty(m, dtype=torch.float16, device="cuda") for _ in range(n)]
    ag_out = [torch.empty(w.count, dtype=torch.float16, device="cuda") for _ in range(n)]
    comm = dcc.Comm(n)
    try:
        comm.register_all("input", xs)
        comm.register_all("output", rs_out)
        comm.register_all("output", ag_out)
        comm.reduce_scatter(xs, rs_out)
        assert comm.check() == dcc.DCC_OK
        host = [W.to_storage(x) for x in xs]
        for r in range(n):
            assert same(W.to_storage(rs_out[r]), oracle.reduce_scatter(host, "fp16", r, m), "fp16"), r
        comm.allgather(rs_out, ag_out)
        assert comm.check() == dcc.DCC_OK
        ag_expect = oracle.allgather([W.to_storage(t) for t in rs_out], "fp16")
        for r in range(n):
            assert np.array_equal(W.to_storage(ag_out[r]), ag_expect), r
        # AG(RS(x)) is the AllReduce
        ar = oracle.allreduce(host, "fp16", nthreads=16)
        assert np.array_equal(ag_expect, ar)
    finally:
        comm.close()


@pytest.mark.parametrize("n,count", [(2, 1), (3, 5), (8, 1000), (8, 1001), (5, 77777), (16, 4096),
                                     (8, 40960), (3, 50000), (2, 262144 + 8)])
@pytest.mark.parametrize("dtype", ["int32", "fp32", "fp16", "bf16"])
def test_reduce_scatter_allgather_ragged(dcc, n, count, dtype):
    """Shards that do not start on 16-byte boundaries take the element path."""
    w = W.with_count(RECIPES[dtype], count * n, n_ranks=n)
    xs = [x.cuda() for x in W.rank_inputs(w)]
    rs_out = [torch.empty(count, dtype=xs[0].dtype, device="cuda") for _ in range(n)]
    ag_out = [torch.empty(count * n, dtype=xs[0].dtype, device="cuda") for _ in range(n)]
    comm = dcc.Comm(n)
    try:
        comm.register_all("input", xs)
        comm.register_all("output", rs_out)
        comm.register_all("output", ag_out)
        comm.reduce_scatter(xs, rs_out)
        comm.allgather(rs_out, ag_out)
        assert comm.check() == dcc.DCC_OK
        host = [W.to_storage(x) for x in xs]
        full = oracle.allreduce(host, dtype)
        for r in range(n):
            assert same(W.to_storage(rs_out[r]), full[r * count:(r + 1) * count], dtype)
            assert same(W.to_storage(ag_out[r]), full, dtype)
    finally:
        comm.close()


def test_random_rs_ag_configurations_match_oracle(dcc, monkeypatch):
    """A hundred seeded random mixes of rank count, per-rank element count (16-byte
    vector path and element path), dtype, CTAs per rank, threads per CTA and the
    entry barrier for the ReduceScatter followed by the AllGather."""
    rng = np.random.default_rng(77)
    for case in range(100):
        n = int(rng.choice([1, 2, 3, 4, 5, 8, 9, 16]))
        dtype = str(rng.choice(sorted(RECIPES)))
        m = int(rng.integers(1, 9000))
        blocks = int(rng.choice([0, 1, 5, 128]))
        threads = int(rng.choice([0, 64, 160, 512]))
        entry_barrier = bool(rng.integers(0, 3) == 0)
        if threads:
            monkeypatch.setenv("DCC_THREADS", str(threads))
        else:
            monkeypatch.delenv("DCC_THREADS", raising=False)
        w = W.with_count(RECIPES[dtype], m * n, n_ranks=n)
        host = W.rank_inputs(w)
        xs = [x.cuda() for x in host]
        rs = [torch.empty(m, dtype=xs[0].dtype, device="cuda") for _ in range(n)]
        ag = [torch.empty(m * n, dtype=xs[0].dtype, device="cuda") for _ in range(n)]
        with dcc.Comm(n) as comm:
            comm.register_all("input", xs)
            comm.register_all("output", rs)
            comm.register_all("output", ag)
            dcc.dcc_set_blocks_per_rank(comm.handle, blocks)
            dcc.dcc_set_entry_barrier(comm.handle, entry_barrier)
            comm.reduce_scatter(xs, rs)
            comm.allgather(rs, ag)
            assert comm.check() == dcc.DCC_OK
        full = oracle.allreduce([W.to_storage(x) for x in host], dtype)
        what = (case, n, dtype, m, blocks, threads, entry_barrier)
        for r in range(n):
            assert same(W.to_storage(rs[r]), full[r * m:(r + 1) * m], dtype), (what, r)
            assert same(W.to_storage(ag[r]), full, dtype), (what, r)


# ---------------------------------------------------------------- synchronisation
@pytest.mark.parametrize("transport", ["default", "l2"])
@pytest.mark.parametrize("n", [1, 2, 3, 8, 16])
def test_ring_barrier_counts(dcc, n, transport, monkeypatch):
    """10^4 iterations: every channel's signal counter and waiter count equal the
    oracle's; up to 8 ranks the default runs the ranks as one cluster (the
    counters are added at the end), "l2" forces the global-memory semaphores."""
    if transport == "l2":
        monkeypatch.setenv("DCC_RING_CLUSTER", "0")
    iters = W.BARRIER_ITERS
    comm = dcc.Comm(n, connect="ring")
    try:
        comm.ring_barrier(iters)
        assert comm.check() == dcc.DCC_OK
        inbound, expected = dcc.dcc_comm_read_semaphores(comm.handle, n)
        ref = oracle.ring_barrier_counts(n, iters)
        assert np.array_equal(inbound, ref)
        assert np.array_equal(expected, ref)
        comm.ring_barrier(3)
        assert comm.check() == dcc.DCC_OK
        inbound, _ = dcc.dcc_comm_read_semaphores(comm.handle, n)
        assert np.array_equal(inbound, oracle.ring_barrier_counts(n, iters + 3))
    finally:
        comm.close()


def test_put_get_and_signal(dcc):
    n = 4
    comm = dcc.Comm(n)
    try:
        ins = [torch.arange(4096, dtype=torch.int32, device="cuda") + 10000 * r for r in range(n)]
        outs = [torch.full((4096,), -1, dtype=torch.int32, device="cuda") for _ in range(n)]
        comm.register_all("input", ins)
        comm.register_all("output", outs)
        # put 1 KiB from rank 1's input (offset 256 B) into rank 3's output (offset 512 B), signalled
        dcc.dcc_channel_put(comm.handle, 1, 3, 512, 256, 1024, signal=True)
        assert comm.check() == dcc.DCC_OK
        got = outs[3].cpu().numpy()
        assert np.array_equal(got[128:384], ins[1].cpu().numpy()[64:320])
        assert np.all(got[:128] == -1) and np.all(got[384:] == -1)
        inbound, expected = dcc.dcc_comm_read_semaphores(comm.handle, n)
        assert inbound[3, 1] == 1 and expected[3, 1] == 1 and inbound.sum() == 1
        # get: rank 0's output [0, 4 KiB) <- rank 2's input [8 KiB, 12 KiB)
        dcc.dcc_channel_get(comm.handle, 0, 2, 8192, 0, 4096)
        assert comm.check() == dcc.DCC_OK
        assert np.array_equal(outs[0].cpu().numpy()[:1024], ins[2].cpu().numpy()[2048:3072])
    finally:
        comm.close()


def test_repeated_calls_never_need_a_reset(dcc):
    """10^4 back-to-back collectives that synchronise through semaphores
    (in-place one-shot, two-shot via scratch) plus barriers, no reset."""
    n, count = 8, 4096 + 3
    w = W.with_count(W.C2, count)
    xs = W.rank_inputs(w)
    arena = Arena(dcc, n, count)
    try:
        send = arena.view(arena.inp, "int32", count)
        recv = arena.view(arena.out, "int32", count)
        for r in range(n):
            send[r].copy_(xs[r])
        h = arena.comm.handle
        for i in range(5000):
            dcc.dcc_allreduce(h, send, recv, count, "int32", "two_shot_scratch")
            dcc.dcc_allreduce(h, recv, recv, count, "int32", "one_shot")
            dcc.dcc_allreduce(h, send, recv, count, "int32", "one_shot_ll")
            dcc.dcc_allreduce(h, recv, recv, count, "int32", "one_shot_ll")
        dcc.dcc_ring_barrier(h, 100)
        assert arena.comm.check() == dcc.DCC_OK
        # recv = 8 * sum(x) after each group; it is recomputed from send every time
        expect = oracle.allreduce([W.to_storage(x) for x in xs], "int32").astype(np.int64) * n
        expect = ((expect + 2 ** 31) % 2 ** 32 - 2 ** 31).astype(np.int32)
        for r in range(n):
            assert np.array_equal(W.to_storage(recv[r]), expect)
        inbound, expected = dcc.dcc_comm_read_semaphores(h, n, block=0)
        assert np.array_equal(inbound, expected)
    finally:
        arena.close()


def test_graph_replay_keeps_epochs(dcc):
    """Collectives captured once into a CUDA graph and replayed: the waits
    count in device memory, so every replay synchronises correctly."""
    n, count = 8, 20000 + 1
    w = W.with_count(W.C4, count)
    xs = W.rank_inputs(w)
    expect = oracle.allreduce([W.to_storage(x) for x in xs], "bf16")
    arena = Arena(dcc, n, count)
    try:
        send = arena.view(arena.inp, "bf16", count)
        recv = arena.view(arena.out, "bf16", count)
        for r in range(n):
            send[r].copy_(xs[r])
        h = arena.comm.handle
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dcc.dcc_allreduce(h, send, recv, count, "bf16", "two_shot_scratch", stream=s)
            dcc.dcc_allreduce(h, send, recv, count, "bf16", "one_shot", stream=s)
            dcc.dcc_allreduce(h, send, recv, count, "bf16", "two_shot", stream=s)
            dcc.dcc_allreduce(h, send, recv, count, "bf16", "two_shot_bulk", stream=s)
            dcc.dcc_allreduce(h, send, recv, count, "bf16", "one_shot_ll", stream=s)
        for _ in range(200):
            g.replay()
        torch.cuda.synchronize()
        assert arena.comm.check() == dcc.DCC_OK
        for r in range(n):
            assert same(W.to_storage(recv[r]), expect, "bf16")
    finally:
        arena.close()


def test_graph_replay_of_rs_ag_fused_and_entry_barrier(dcc):
    """ReduceScatter, AllGather (plain and through the entry barrier) and both
    fused linear-layer kernels captured into one CUDA graph and replayed: the
    same bits as the oracle after every replay."""
    n, m = 8, 4104
    g = torch.Generator().manual_seed(11)
    xs = [torch.randn(n * m, generator=g).to(torch.bfloat16).cuda() for _ in range(n)]
    rs = [torch.empty(m, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    ag = [torch.empty(n * m, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    rs_eb = [torch.empty_like(t) for t in rs]
    ag_eb = [torch.empty_like(t) for t in ag]
    rows = 64
    lin = {}
    for kp in (1024, 4096):  # thread-load kernel and bulk-copy kernel
        ws = [torch.randint(-3, 4, (rows * kp,), generator=g).to(torch.bfloat16).cuda() for _ in range(n)]
        xv = [torch.randint(-3, 4, (kp,), generator=g).to(torch.bfloat16).cuda() for _ in range(n)]
        yv = [torch.empty(rows, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        lin[kp] = (ws, xv, yv)
    host = [W.to_storage(x.cpu()) for x in xs]
    full = oracle.allreduce(host, "bf16")
    with dcc.Comm(n) as comm, dcc.Comm(n) as comm_eb:
        for c, (r_, a_) in ((comm, (rs, ag)), (comm_eb, (rs_eb, ag_eb))):
            c.register_all("input", xs)
            c.register_all("output", r_)
            c.register_all("output", a_)
        for ws, xv, yv in lin.values():
            comm.register_all("input", ws)
            comm.register_all("input", xv)
            comm.register_all("output", yv)
        dcc.dcc_set_entry_barrier(comm_eb.handle, True)
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            dcc.dcc_reduce_scatter(comm.handle, xs, rs, m, "bf16", stream=s)
            dcc.dcc_allgather(comm.handle, rs, ag, m, "bf16", stream=s)
            dcc.dcc_reduce_scatter(comm_eb.handle, xs, rs_eb, m, "bf16", stream=s)
            dcc.dcc_allgather(comm_eb.handle, rs_eb, ag_eb, m, "bf16", stream=s)
            for kp, (ws, xv, yv) in lin.items():
                dcc.dcc_linear_allreduce(comm.handle, ws, xv, yv, rows, kp, "bf16", stream=s)
        for _ in range(50):
            graph.replay()
        torch.cuda.synchronize()
        assert comm.check() == dcc.DCC_OK and comm_eb.check() == dcc.DCC_OK
    for r in range(n):
        for got_rs, got_ag in ((rs, ag), (rs_eb, ag_eb)):
            assert same(W.to_storage(got_rs[r]), full[r * m:(r + 1) * m], "bf16")
            assert same(W.to_storage(got_ag[r]), full, "bf16")
    for kp, (ws, xv, yv) in lin.items():
        expect = oracle.linear_allreduce([W.to_storage(w.cpu()) for w in ws], [W.to_storage(x.cpu()) for x in xv],
                                         "bf16", rows, kp)
        for r in range(n):
            assert np.array_equal(W.to_storage(yv[r]), expect), (kp, r)


def test_concurrent_streams(dcc):
    """Kernels that never wait overlap freely on one communicator (two streams,
    two-shot push and ReduceScatter/AllGather on separate buffers), and two
    communicators run their synchronising kernels (in-place one-shot, two-shot
    via scratch) on two streams at the same time: every result as the oracle's."""
    n, count = 8, 3 * 4096 + 24
    g = torch.Generator().manual_seed(21)
    host = [torch.randint(-8, 9, (count,), generator=g).float() for _ in range(n)]
    expect = oracle.allreduce([W.to_storage(h) for h in host], "fp32")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def bufs():
        return [h.cuda() for h in host], [torch.empty(count, device="cuda") for _ in range(n)]

    # one communicator, two streams, wait-free kernels on disjoint buffers
    (xa, ya), (xb, yb) = bufs(), bufs()
    m = count // n
    rs = [torch.empty(m, device="cuda") for _ in range(n)]
    ag = [torch.empty(m * n, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        for t in (xa, xb):
            comm.register_all("input", t)
        for t in (ya, yb, rs, ag):
            comm.register_all("output", t)
        torch.cuda.synchronize()
        for _ in range(20):
            dcc.dcc_allreduce(comm.handle, xa, ya, count, "fp32", "two_shot", stream=s1)
            dcc.dcc_reduce_scatter(comm.handle, xb, rs, m, "fp32", stream=s2)
            dcc.dcc_allgather(comm.handle, rs, ag, m, "fp32", stream=s2)
        torch.cuda.synchronize()
        assert comm.check() == dcc.DCC_OK
    for r in range(n):
        assert same(W.to_storage(ya[r]), expect, "fp32")
        assert same(W.to_storage(ag[r]), expect[: m * n], "fp32")
    # two communicators, two streams, synchronising kernels at the same time:
    # a ring barrier then an in-place one-shot on one, two-shots via scratch on
    # the other (neither waits on the other's semaphores)
    (xc, _), (xd, yd) = bufs(), bufs()
    scr = [torch.empty(count, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as c1, dcc.Comm(n) as c2:
        c1.register_all("input", xc)
        c2.register_all("input", xd)
        c2.register_all("output", yd)
        c2.register_all("scratch", scr)
        torch.cuda.synchronize()
        c1.ring_barrier(2000, stream=s1)
        dcc.dcc_allreduce(c1.handle, xc, xc, count, "fp32", "one_shot", stream=s1)
        for _ in range(20):
            dcc.dcc_allreduce(c2.handle, xd, yd, count, "fp32", "two_shot_scratch", stream=s2)
        torch.cuda.synchronize()
        assert c1.check() == dcc.DCC_OK and c2.check() == dcc.DCC_OK
        inbound, expected = dcc.dcc_comm_read_semaphores(c1.handle, n)
        assert np.array_equal(inbound, expected)
    for r in range(n):
        assert same(W.to_storage(xc[r]), expect, "fp32")
        assert same(W.to_storage(yd[r]), expect, "fp32")


@pytest.mark.parametrize("transport", ["default", "l2"])
def test_lost_signal_times_out_cleanly(dcc, transport, monkeypatch):
    """A rank that never signals makes its peers' waits run out: the kernel
    records DCC_ERR_TIMEOUT and returns; the GPU stays usable (the ring barrier
    through a cluster's shared memory and through the global semaphores)."""
    if transport == "l2":
        monkeypatch.setenv("DCC_RING_CLUSTER", "0")
    n = 4
    comm = dcc.Comm(n, connect="all")
    try:
        dcc.dcc_set_wait_timeout_us(comm.handle, 50000)
        dcc.dcc_debug_skip_signal(comm.handle, 1)
        comm.ring_barrier(10)
        assert comm.check() == dcc.DCC_ERR_TIMEOUT
        # once rank 1's signal is lost every rank ends up waiting on its ring
        # predecessor; whichever wait gives up first records itself
        rank, peer, block = dcc.dcc_comm_error_detail(comm.handle)
        assert 0 <= rank < n and (rank - peer) % n == 1 and block == 0
        with pytest.raises(dcc.DccError) as e:
            comm.ring_barrier(1)
        assert e.value.code == dcc.DCC_ERR_TIMEOUT
    finally:
        comm.close()
    # the same for a collective that synchronises through every channel
    comm = dcc.Comm(n)
    try:
        count = 100000
        bufs = [torch.ones(count, dtype=torch.float32, device="cuda") for _ in range(n)]
        scr = [torch.empty(count, dtype=torch.float32, device="cuda") for _ in range(n)]
        comm.register_all("input", bufs)
        comm.register_all("scratch", scr)
        dcc.dcc_set_wait_timeout_us(comm.handle, 50000)
        dcc.dcc_debug_skip_signal(comm.handle, 3)
        comm.allreduce(bufs, bufs, algo="two_shot_scratch")
        assert comm.check() == dcc.DCC_ERR_TIMEOUT
        assert dcc.dcc_comm_error_detail(comm.handle)[1] == 3
    finally:
        comm.close()
    # a fresh communicator works
    with dcc.Comm(2) as c2:
        a = [torch.ones(1000, device="cuda") for _ in range(2)]
        c2.register_all("input", a)
        c2.allreduce(a, a, algo="one_shot")
        assert c2.check() == dcc.DCC_OK
        assert torch.all(a[0] == 2)


# ---------------------------------------------------------------- beyond 32-bit element indices
def test_more_than_2_31_elements_per_rank(dcc):
    """4 GiB + 26 bytes of bf16 per rank (2^31 + 13 elements): 64-bit index
    arithmetic on the device and in the launch shapes.  Sampled windows (random
    ones, both sides of element 2^31 and the ragged tail) are checked against
    the oracle run on those elements.  Inputs are filled and outputs cleared
    in 2^24-element slices, and samples are read back as contiguous slices, so
    every torch operation stays small."""
    n, count, chunk = 2, 2 ** 31 + 13, 2 ** 24
    free, _ = torch.cuda.mem_get_info()
    if free < 24 * 2 ** 30:
        pytest.skip("needs 24 GiB of free device memory")
    pat = ((torch.arange(chunk, device="cuda") % 251) - 125).to(torch.bfloat16)
    xs = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    for r, x in enumerate(xs):
        src = pat * (r + 1)
        for a in range(0, count, chunk):
            b = min(count, a + chunk)
            x[a:b].copy_(src[: b - a])
    ys = [torch.empty_like(x) for x in xs]

    def clear(t):
        for a in range(0, count, chunk):
            t[a: min(count, a + chunk)].zero_()

    rng = np.random.default_rng(5)
    windows = [(int(o), 64) for o in np.sort(rng.integers(0, count - 64, 48))]
    windows += [(2 ** 31 - 64, count - (2 ** 31 - 64)), (count - 40, 40)]  # up to the last element
    assert all(0 <= o and o + k <= count for o, k in windows)

    def sample(t):
        return np.concatenate([W.to_storage(t[o: o + k].cpu()) for o, k in windows])

    expect = oracle.allreduce([sample(x) for x in xs], "bf16")
    with dcc.Comm(n) as comm:
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        for algo in ("one_shot", "two_shot"):
            for y in ys:
                clear(y)
            comm.allreduce(xs, ys, algo=algo)
            assert comm.check() == dcc.DCC_OK
            for r in range(n):
                assert same(sample(ys[r]), expect, "bf16"), (algo, r)
        # in place through the two-shot push
        comm.allreduce(xs, xs, algo="two_shot")
        assert comm.check() == dcc.DCC_OK
        for r in range(n):
            assert same(sample(xs[r]), expect, "bf16"), ("in place", r)
    del xs, ys
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- entry barrier
@pytest.mark.parametrize("n", [2, 5, 8, 16])
def test_entry_barrier_same_bits_and_counts(dcc, n):
    """With the entry barrier on, every thread-copy AllReduce, the ReduceScatter
    and the AllGather return the oracle's bits, and each launch adds exactly one
    signal from every rank to every other rank on every block slot it used."""
    count = 8 * n * 1000 + 3 * n  # ragged: several vectors per shard plus a tail
    w = W.with_count(W.C4, count, n_ranks=n)
    xs = W.rank_inputs(w)
    expect = oracle.allreduce([W.to_storage(x) for x in xs], "bf16")
    arena = Arena(dcc, n, count)
    try:
        h = arena.comm.handle
        dcc.dcc_set_entry_barrier(h, True)
        before, _ = dcc.dcc_comm_read_semaphores(h, n, block=0)
        launches = 0
        for algo in ("one_shot", "two_shot", "two_shot_scratch"):
            for inplace in (False, True):
                outs = run_allreduce(dcc, arena, xs, "bf16", algo, inplace)
                launches += 1
                assert all(same(o, expect, "bf16") for o in outs), (algo, inplace)
        # block slot 0 took part in every launch: one entry signal per ordered pair each,
        # plus the scratch kernel's phase barrier and the in-place one-shot's chunk barriers
        after, expected = dcc.dcc_comm_read_semaphores(h, n, block=0)
        off = ~np.eye(n, dtype=bool)
        assert np.all(after[off] - before[off] >= launches)
        assert np.array_equal(after, expected)  # every signal was waited for
        # bulk and LL have no entry barrier
        send = arena.view(arena.inp, "bf16", count)
        for algo in ("two_shot_bulk", "one_shot_ll"):
            with pytest.raises(dcc.DccError) as e:
                dcc.dcc_allreduce(h, send, send, count, "bf16", algo)
            assert e.value.code == dcc.DCC_ERR_UNSUPPORTED
        assert arena.comm.check() == dcc.DCC_OK
    finally:
        arena.close()
    # ReduceScatter and AllGather through the entry barrier
    m = count // n
    rs_in = [x[: m * n].cuda() for x in xs]
    rs_out = [torch.empty(m, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    ag_out = [torch.empty(m * n, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", rs_in)
        comm.register_all("output", rs_out)
        comm.register_all("output", ag_out)
        dcc.dcc_set_entry_barrier(comm.handle, True)
        b0, _ = dcc.dcc_comm_read_semaphores(comm.handle, n, block=0)
        comm.reduce_scatter(rs_in, rs_out)
        comm.allgather(rs_out, ag_out)
        assert comm.check() == dcc.DCC_OK
        b1, e1 = dcc.dcc_comm_read_semaphores(comm.handle, n, block=0)
        off = ~np.eye(n, dtype=bool)
        assert np.all(b1[off] - b0[off] == 2) and np.array_equal(b1, e1)
        host = [W.to_storage(x.cpu()) for x in rs_in]
        full = oracle.allreduce(host, "bf16")
        for r in range(n):
            assert same(W.to_storage(rs_out[r]), full[r * m:(r + 1) * m], "bf16")
            assert same(W.to_storage(ag_out[r]), full, "bf16")


def test_entry_barrier_lost_signal_times_out(dcc):
    """The two-shot push has no wait of its own; with the entry barrier a rank
    that never signals makes the launch report DCC_ERR_TIMEOUT."""
    n = 4
    comm = dcc.Comm(n)
    try:
        bufs = [torch.ones(50000, dtype=torch.float32, device="cuda") for _ in range(n)]
        comm.register_all("input", bufs)
        dcc.dcc_set_wait_timeout_us(comm.handle, 50000)
        dcc.dcc_set_entry_barrier(comm.handle, True)
        dcc.dcc_debug_skip_signal(comm.handle, 2)
        comm.allreduce(bufs, bufs, algo="two_shot")
        assert comm.check() == dcc.DCC_ERR_TIMEOUT
        assert dcc.dcc_comm_error_detail(comm.handle)[1] == 2
    finally:
        comm.close()


# ---------------------------------------------------------------- host-side errors on a device
def test_argument_errors(dcc):
    n = 2
    comm = dcc.Comm(n, connect="none")
    try:
        h = comm.handle
        a = [torch.zeros(1024, device="cuda") for _ in range(n)]
        b = [torch.zeros(1024, device="cuda") for _ in range(n)]
        E = dcc.DccError

        def code(f, *args, **kw):
            with pytest.raises(E) as e:
                f(*args, **kw)
            return e.value.code

        assert code(dcc.dcc_allreduce, h, a, b, 1024, "fp32") == dcc.DCC_ERR_NOT_REGISTERED
        comm.register_all("input", a)
        comm.register_all("output", b)
        assert code(dcc.dcc_allreduce, h, a, b, 1024, "fp32") == dcc.DCC_ERR_NO_CHANNEL
        dcc.dcc_memory_channel_make(h, 0, 1)
        dcc.dcc_memory_channel_make(h, 1, 0)
        dcc.dcc_memory_channel_make(h, 1, 0)  # idempotent
        dcc.dcc_allreduce(h, a, b, 1024, "fp32")
        assert code(dcc.dcc_allreduce, h, a, b, 1025, "fp32") == dcc.DCC_ERR_NOT_REGISTERED
        mis = [x[1:] for x in a]
        assert code(dcc.dcc_allreduce, h, mis, b, 100, "fp32") == dcc.DCC_ERR_MISALIGNED
        over = [b[0][4:], b[1]]
        assert code(dcc.dcc_allreduce, h, [b[0], b[1]], [b[0][4:], a[1]], 100, "fp32") == \
            dcc.DCC_ERR_INVALID_ARG
        del over
        assert code(dcc.dcc_allreduce, h, a, b, 16, 7) == dcc.DCC_ERR_INVALID_ARG
        assert code(dcc.dcc_allreduce, h, a, b, 16, "fp32", 9) == dcc.DCC_ERR_INVALID_ARG
        assert code(dcc.dcc_allreduce, h, a, b, 16, "fp32", "two_shot_scratch") == \
            dcc.DCC_ERR_NOT_REGISTERED  # no scratch window
        assert code(dcc.dcc_memory_channel_make, h, 0, 0) == dcc.DCC_ERR_INVALID_ARG
        assert code(dcc.dcc_memory_channel_make, h, 0, 2) == dcc.DCC_ERR_INVALID_ARG
        assert code(dcc.dcc_register_buffer, h, 0, "input", a[0][1:], 16) == dcc.DCC_ERR_MISALIGNED
        assert code(dcc.dcc_register_buffer, h, 2, "input", a[0]) == dcc.DCC_ERR_INVALID_ARG
        assert code(dcc.dcc_ring_barrier, h, -1) == dcc.DCC_ERR_INVALID_ARG
        dcc.dcc_allreduce(h, a, b, 0, "fp32")  # empty: no-op
        # RS/AG with overlapping ranges are rejected
        assert code(dcc.dcc_reduce_scatter, h, a, [a[0][:256], a[1][:256]], 256, "fp32") == \
            dcc.DCC_ERR_INVALID_ARG
        assert comm.check() == dcc.DCC_OK
    finally:
        comm.close()


@pytest.mark.parametrize("mode", ["zero_copy", "staged", "pageable"])
@pytest.mark.parametrize("count,inplace", [(300001, False), (3 * 4194304 + 13, False),
                                           (2 * 4194304 + 8, True)])
def test_allreduce_from_host(dcc, count, inplace, mode, monkeypatch):
    """Host buffers in, host buffers out: zero copy over the host link (pinned
    buffers), or staged through device buffers and pipelined in 8 MiB-per-rank
    chunks (forced, or because the host memory is pageable); one chunk, three
    chunks with a ragged last one, in-place staging."""
    n = 8
    if mode == "staged":
        monkeypatch.setenv("DCC_ZERO_COPY", "0")
    w = W.with_count(W.C4, count)
    if mode == "pageable":
        xs = [x.clone() for x in W.rank_inputs(w)]
        outs = [torch.empty_like(x) for x in xs]
    else:
        xs = [x.pin_memory() for x in W.rank_inputs(w)]
        outs = [torch.empty_like(x).pin_memory() for x in xs]
    dev_in = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    dev_out = dev_in if inplace else [torch.empty_like(d) for d in dev_in]
    comm = dcc.Comm(n)
    try:
        comm.register_all("input", dev_in)
        if not inplace:
            comm.register_all("output", dev_out)
        s = torch.cuda.Stream()
        for _ in range(2):  # twice: the second call reuses the pipeline's streams and events
            for o in outs:
                o.zero_()
            dcc.dcc_allreduce_from_host(comm.handle, xs, outs, dev_in, dev_out, count, "bf16",
                                        stream=s)
            assert comm.check(s) == dcc.DCC_OK
            expect = oracle.allreduce([W.to_storage(x) for x in xs], "bf16", nthreads=8)
            for o in outs:
                assert same(W.to_storage(o), expect, "bf16")
    finally:
        comm.close()


def test_auto_selection(dcc):
    """AUTO follows the measured crossover table (the tuning JSON) for every
    rank count and dtype, and a per-communicator override moves it."""
    from driven_collective_communication_gb300 import build
    table = build.load_auto_table()
    for n in (1, 2, 3, 4, 5, 8, 12, 16):
        with dcc.Comm(n) as c:
            for t, eb in (("int32", 4), ("fp32", 4), ("fp16", 2), ("bf16", 2)):
                lim = table[n][t] // eb  # elements
                if lim:
                    assert dcc.dcc_select_algo(c.handle, lim, t) == "one_shot", (n, t)
                assert dcc.dcc_select_algo(c.handle, lim + 1, t) == "two_shot", (n, t)
    with dcc.Comm(8) as c:
        dcc.dcc_set_algo_threshold(c.handle, "bf16", 65536)
        assert dcc.dcc_select_algo(c.handle, 32768, "bf16") == "one_shot"
        assert dcc.dcc_select_algo(c.handle, 32769, "bf16") == "two_shot"
        # streaming two-shot: one 16-byte vector per thread over the shard
        b, t = dcc.dcc_launch_shape(c.handle, W.C4.count, "bf16", "two_shot")
        assert b * t >= W.C4.count // 8 // 8 and t > 0
        # a kernel that synchronises ranks stays within one wave and its slots
        b, t = dcc.dcc_launch_shape(c.handle, W.C4.count, "bf16", "two_shot_scratch")
        assert 1 <= b <= dcc.DCC_MAX_BLOCKS_PER_RANK and t > 0
