"""GPU parity of the MAX / MIN AllReduce and ReduceScatter against the CPU oracle.

MAX / MIN return one input's bits (or the canonical quiet NaN), so the
comparison is bit for bit, NaN bits included.  Inputs are seeded raw bit
patterns with NaN, infinities, signed zeros and subnormals mixed in, and
values copied between ranks so that ties (equal values, +0 against -0) occur.
"""
import numpy as np
import pytest
import torch

import oracle
from driven_collective_communication_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DTYPES = ("int32", "fp32", "fp16", "bf16")
OPS = ("max", "min")
RAW = {"int32": np.int32, "fp32": np.uint32, "fp16": np.uint16, "bf16": np.uint16}
SPECIALS = {
    "fp32": [0x00000000, 0x80000000, 0x7f800000, 0xff800000, 0x7fc00000, 0xffc00001, 0x00000001,
             0x80000001, 0x3f800000, 0xbf800000, 0x7f7fffff, 0xff7fffff],
    "fp16": [0x0000, 0x8000, 0x7c00, 0xfc00, 0x7e00, 0xfe01, 0x0001, 0x8001, 0x3c00, 0xbc00, 0x7bff, 0xfbff],
    "bf16": [0x0000, 0x8000, 0x7f80, 0xff80, 0x7fc0, 0xffc1, 0x0001, 0x8001, 0x3f80, 0xbf80, 0x7f7f, 0xff7f],
    "int32": [0, -1, 1, 2 ** 31 - 1, -2 ** 31, 7, -7],
}


@pytest.fixture(scope="module")
def dcc():
    from driven_collective_communication_gb300 import build
    build.build()
    from driven_collective_communication_gb300 import dcc as mod
    torch.cuda.set_device(0)
    return mod


def raw_inputs(seed, dtype, n, count):
    """n rank inputs of `count` raw elements (storage dtype of the oracle):
    random bit patterns, a quarter replaced by special values, a quarter by the
    same element of rank 0 (ties)."""
    rng = np.random.default_rng(seed)
    bits = 32 if dtype in ("int32", "fp32") else 16
    xs = []
    for r in range(n):
        x = rng.integers(0, 2 ** bits, size=count, dtype=np.uint64).astype(np.uint32 if bits == 32 else np.uint16)
        if dtype == "int32":
            x = x.view(np.int32)
        sp = np.array(SPECIALS[dtype], dtype=np.int64)
        pick = rng.random(count) < 0.25
        x[pick] = sp[rng.integers(0, len(sp), size=int(pick.sum()))].astype(x.dtype)
        if r > 0:
            tie = rng.random(count) < 0.25
            x[tie] = xs[0][tie]
        xs.append(x)
    return [x.view(oracle.STORAGE[dtype]) for x in xs]


def to_device(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int32 if a.dtype.itemsize == 4 else np.int16).copy())
    return t.view(W.TORCH_DTYPES[dtype]).cuda()


def to_host_bits(t, dtype):
    raw = t.view(torch.int32 if W.ELEM_BYTES[dtype] == 4 else torch.int16).cpu().numpy()
    return raw.view(RAW[dtype])


def bits_equal(got_t, expect, dtype):
    return np.array_equal(to_host_bits(got_t, dtype), np.asarray(expect).view(RAW[dtype]))


class Arena:
    def __init__(self, dcc, n, bytes_per_rank):
        self.n = n
        self.comm = dcc.Comm(n)
        nb = bytes_per_rank + 4096
        self.inp = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(n)]
        self.out = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(n)]
        for r in range(n):
            self.comm.register(r, "input", self.inp[r])
            self.comm.register(r, "output", self.out[r])

    def view(self, bufs, dtype, count):
        eb = W.ELEM_BYTES[dtype]
        assert count * eb <= bufs[0].numel()
        return [b[: count * eb].view(W.TORCH_DTYPES[dtype]) for b in bufs]

    def close(self):
        self.comm.close()


def run_op(dcc, arena, xs, dtype, op, algo, inplace):
    count = len(xs[0])
    send = arena.view(arena.inp, dtype, count)
    for r in range(arena.n):
        send[r].copy_(to_device(xs[r], dtype))
    recv = send if inplace else arena.view(arena.out, dtype, count)
    if not inplace:
        for r in range(arena.n):
            recv[r].zero_()
    dcc.dcc_allreduce_op(arena.comm.handle, send, recv, count, dtype, op, algo)
    rc = arena.comm.check()
    assert rc == dcc.DCC_OK, dcc.dcc_error_string(rc)
    return recv


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16])
def test_allreduce_op_parity_sweep(dcc, n):
    """MAX and MIN, every dtype, one-shot / two-shot / AUTO, in and out of place,
    counts from one element to several CTAs' worth with a ragged tail, against
    the oracle bit for bit (compile-time and runtime-N instances)."""
    counts = [1, 5, 8, 16 * n + 3, 3 * 512 * 8 + 5, 70001]
    arena = Arena(dcc, n, max(counts) * 4)
    try:
        for dtype in DTYPES:
            for count in counts:
                xs = raw_inputs(1000 * n + count, dtype, n, count)
                for op in OPS:
                    expect = oracle.allreduce_op(xs, dtype, op)
                    for algo in ("auto", "one_shot", "two_shot"):
                        for inplace in (False, True):
                            outs = run_op(dcc, arena, xs, dtype, op, algo, inplace)
                            for r in range(n):
                                assert bits_equal(outs[r], expect, dtype), (dtype, count, op, algo, inplace, r)
    finally:
        arena.close()


@pytest.mark.parametrize("n", [2, 3, 8])
def test_reduce_scatter_op_parity(dcc, n):
    """MAX / MIN ReduceScatter: vector path (shards on 16-byte boundaries) and
    scalar path (ragged shards), every dtype, against the oracle."""
    recv_counts = [1, 7, 8, 1000, 4099, 20000]
    arena = Arena(dcc, n, max(recv_counts) * n * 4)
    try:
        for dtype in DTYPES:
            for m in recv_counts:
                xs = raw_inputs(77 * n + m, dtype, n, m * n)
                send = arena.view(arena.inp, dtype, m * n)
                recv = arena.view(arena.out, dtype, m)
                for r in range(n):
                    send[r].copy_(to_device(xs[r], dtype))
                for op in OPS:
                    expect = oracle.allreduce_op(xs, dtype, op)
                    for r in range(n):
                        recv[r].zero_()
                    dcc.dcc_reduce_scatter_op(arena.comm.handle, send, recv, m, dtype, op)
                    assert arena.comm.check() == dcc.DCC_OK
                    for r in range(n):
                        assert bits_equal(recv[r], expect[r * m:(r + 1) * m], dtype), (dtype, m, op, r)
    finally:
        arena.close()


def test_sum_through_op_entry_points_matches_plain_calls(dcc):
    """DCC_OP_SUM through dcc_allreduce_op / dcc_reduce_scatter_op is the plain
    sum collective."""
    n, count = 4, 4099
    w = W.with_count(W.C4, count, n_ranks=n)
    xs = [x.cuda() for x in W.rank_inputs(w)]
    with dcc.Comm(n) as comm:
        ys = [torch.empty_like(x) for x in xs]
        zs = [torch.empty_like(x) for x in xs]
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        comm.register_all("output", zs)
        comm.allreduce(xs, ys)
        comm.allreduce_op(xs, zs, op="sum")
        assert comm.check() == dcc.DCC_OK
        for r in range(n):
            assert torch.equal(ys[r].view(torch.int16), zs[r].view(torch.int16))
        m = count // n
        rs_a = [torch.empty(m, dtype=xs[0].dtype, device="cuda") for _ in range(n)]
        rs_b = [torch.empty(m, dtype=xs[0].dtype, device="cuda") for _ in range(n)]
        comm.register_all("output", rs_a)
        comm.register_all("output", rs_b)
        dcc.dcc_reduce_scatter(comm.handle, xs, rs_a, m, "bf16")
        dcc.dcc_reduce_scatter_op(comm.handle, xs, rs_b, m, "bf16", "sum")
        assert comm.check() == dcc.DCC_OK
        for r in range(n):
            assert torch.equal(rs_a[r].view(torch.int16), rs_b[r].view(torch.int16))


def test_op_argument_errors(dcc):
    """Schedules without MAX / MIN instances return DCC_ERR_UNSUPPORTED; an op
    code outside the enum is DCC_ERR_INVALID_ARG; nothing is written."""
    n, count = 4, 1024
    xs = [torch.full((count,), float(r), device="cuda") for r in range(n)]
    ys = [torch.full((count,), -5.0, device="cuda") for _ in range(n)]
    scr = [torch.empty(count, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        comm.register_all("scratch", scr)
        for algo in ("two_shot_scratch", "two_shot_bulk", "one_shot_ll"):
            with pytest.raises(dcc.DccError) as e:
                dcc.dcc_allreduce_op(comm.handle, xs, ys, count, "fp32", "max", algo)
            assert e.value.code == dcc.DCC_ERR_UNSUPPORTED
        for bad in (3, -1):
            with pytest.raises(dcc.DccError) as e:
                dcc.dcc_allreduce_op(comm.handle, xs, ys, count, "fp32", bad)
            assert e.value.code == dcc.DCC_ERR_INVALID_ARG
            with pytest.raises(dcc.DccError) as e:
                dcc.dcc_reduce_scatter_op(comm.handle, xs, ys, count // n, "fp32", bad)
            assert e.value.code == dcc.DCC_ERR_INVALID_ARG
        assert comm.check() == dcc.DCC_OK
    torch.cuda.synchronize()
    for y in ys:
        assert torch.all(y == -5.0)


@pytest.mark.parametrize("n", [5, 8])
def test_op_with_entry_barrier(dcc, n):
    """With the entry barrier on, MAX / MIN run on the barrier (runtime-N)
    instances, cooperatively; results unchanged."""
    count = 3 * 4096 + 9
    arena = Arena(dcc, n, count * 4)
    try:
        dcc.dcc_set_entry_barrier(arena.comm.handle, True)
        for dtype in ("fp32", "bf16"):
            xs = raw_inputs(5 + n, dtype, n, count)
            for op in OPS:
                expect = oracle.allreduce_op(xs, dtype, op)
                for algo in ("one_shot", "two_shot"):
                    for inplace in (False, True):
                        outs = run_op(dcc, arena, xs, dtype, op, algo, inplace)
                        for r in range(n):
                            assert bits_equal(outs[r], expect, dtype), (dtype, op, algo, inplace, r)
                m = count // n
                send = arena.view(arena.inp, dtype, m * n)
                recv = arena.view(arena.out, dtype, m)
                for r in range(n):
                    send[r].copy_(to_device(xs[r][: m * n], dtype))
                dcc.dcc_reduce_scatter_op(arena.comm.handle, send, recv, m, dtype, op)
                assert arena.comm.check() == dcc.DCC_OK
                full = oracle.allreduce_op([x[: m * n] for x in xs], dtype, op)
                for r in range(n):
                    assert bits_equal(recv[r], full[r * m:(r + 1) * m], dtype)
    finally:
        arena.close()


def test_op_full_size(dcc):
    """8 ranks x 256 MiB bf16 (the sum benchmark's size), MAX and MIN through
    AUTO (two-shot at this size), in the launch configuration the library
    picks; every element of every rank's output against the oracle, bit for
    bit (NaN inputs give the canonical NaN on both sides)."""
    n, count = 8, 134217728
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    xs = [torch.randn(count, generator=g, device="cuda").to(torch.bfloat16) for _ in range(n)]
    xs[3][::1000] = float("nan")
    xs[5][7::997] = -0.0
    ys = [torch.empty_like(x) for x in xs]
    host = [to_host_bits(x, "bf16") for x in xs]
    with dcc.Comm(n) as comm:
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        for op in OPS:
            comm.allreduce_op(xs, ys, op=op)
            assert comm.check() == dcc.DCC_OK
            expect = oracle.allreduce_op(host, "bf16", op)
            for r in range(n):
                got = to_host_bits(ys[r], "bf16")
                assert np.array_equal(got, expect), (op, r, int(np.count_nonzero(got != expect)))


def test_random_op_configurations_match_oracle(dcc, monkeypatch):
    """150 seeded random mixes of rank count (compiled and runtime-N
    instances), element count, dtype, MAX / MIN, schedule, in / out of place,
    CTAs per rank, threads per CTA, entry barrier and programmatic dependent
    launch, on raw inputs with specials, each against the oracle bit for bit."""
    rng = np.random.default_rng(4242)
    for case in range(150):
        n = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16]))
        dtype = str(rng.choice(DTYPES))
        count = int(rng.integers(1, 60000))
        op = str(rng.choice(OPS))
        algo = str(rng.choice(["auto", "one_shot", "two_shot"]))
        inplace = bool(rng.integers(0, 2))
        blocks = int(rng.choice([0, 1, 3, 17, 128]))
        threads = int(rng.choice([0, 64, 96, 256]))
        entry_barrier = bool(rng.integers(0, 4) == 0)
        pdl = bool(rng.integers(0, 2))
        if threads:
            monkeypatch.setenv("DCC_THREADS", str(threads))
        else:
            monkeypatch.delenv("DCC_THREADS", raising=False)
        xs = raw_inputs(9000 + case, dtype, n, count)
        expect = oracle.allreduce_op(xs, dtype, op)
        arena = Arena(dcc, n, count * 4)
        try:
            h = arena.comm.handle
            dcc.dcc_set_blocks_per_rank(h, blocks)
            dcc.dcc_set_entry_barrier(h, entry_barrier)
            dcc.dcc_set_pdl(h, pdl)
            outs = run_op(dcc, arena, xs, dtype, op, algo, inplace)
            what = (case, n, dtype, count, op, algo, inplace, blocks, threads, entry_barrier, pdl)
            for r in range(n):
                assert bits_equal(outs[r], expect, dtype), (what, r)
        finally:
            arena.close()


def test_random_op_reduce_scatter_configurations(dcc, monkeypatch):
    """60 seeded random ReduceScatter mixes (rank count, shard size on and off
    16-byte boundaries, dtype, MAX / MIN, CTAs per rank, threads, entry
    barrier, programmatic dependent launch) against the oracle."""
    rng = np.random.default_rng(4343)
    for case in range(60):
        n = int(rng.choice([2, 3, 4, 5, 8, 9, 16]))
        dtype = str(rng.choice(DTYPES))
        m = int(rng.integers(1, 9000))
        op = str(rng.choice(OPS))
        blocks = int(rng.choice([0, 1, 5, 64]))
        threads = int(rng.choice([0, 64, 256]))
        if threads:
            monkeypatch.setenv("DCC_THREADS", str(threads))
        else:
            monkeypatch.delenv("DCC_THREADS", raising=False)
        xs = raw_inputs(7000 + case, dtype, n, m * n)
        expect = oracle.allreduce_op(xs, dtype, op)
        arena = Arena(dcc, n, m * n * 4)
        try:
            h = arena.comm.handle
            dcc.dcc_set_blocks_per_rank(h, blocks)
            dcc.dcc_set_entry_barrier(h, bool(rng.integers(0, 4) == 0))
            dcc.dcc_set_pdl(h, bool(rng.integers(0, 2)))
            send = arena.view(arena.inp, dtype, m * n)
            recv = arena.view(arena.out, dtype, m)
            for r in range(n):
                send[r].copy_(to_device(xs[r], dtype))
                recv[r].zero_()
            dcc.dcc_reduce_scatter_op(h, send, recv, m, dtype, op)
            assert arena.comm.check() == dcc.DCC_OK
            for r in range(n):
                assert bits_equal(recv[r], expect[r * m:(r + 1) * m], dtype), (case, n, dtype, m, op, r)
        finally:
            arena.close()
