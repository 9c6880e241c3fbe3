"""Pins of the CPU oracle against things other than itself.

Closed forms, hand-derived IEEE cases (tests/golden), an independent pure-Python
brute force, exhaustive conversion round trips, conversions of a second library
(torch), the recursive-summation error bound, and the RS/AG/AllReduce identities.
Each test names the mistake it is there to catch.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from driven_collective_communication_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FLOAT_DTYPES = ("fp32", "fp16", "bf16")
ALL_DTYPES = ("int32",) + FLOAT_DTYPES

ONE_BITS = {"fp16": 0x3C00, "bf16": 0x3F80}


def f32_of(x):
    return np.float32(x)


def value_to_storage(v, dtype):
    """Exact encoding of a Python value into raw storage (via torch, a library)."""
    if dtype == "int32":
        return np.int32(v)
    if dtype == "fp32":
        return np.float32(v)
    t = torch.tensor([v], dtype=torch.float64).to(W.TORCH_DTYPES[dtype])
    return W.to_storage(t)[0]


def storage_to_float(a, dtype):
    """Raw storage -> float64 numpy via torch's widening (a second library)."""
    if dtype in ("int32", "fp32"):
        return np.asarray(a, dtype=np.float64)
    return W.from_storage(np.asarray(a, dtype=np.uint16), dtype).to(torch.float64).numpy()


def random_raw(rng, dtype, n, specials=False):
    if dtype == "int32":
        return rng.integers(-2 ** 31, 2 ** 31, size=n, dtype=np.int64).astype(np.int32)
    if dtype == "fp32":
        x = (rng.standard_normal(n) * np.exp2(rng.integers(-30, 30, size=n))).astype(np.float32)
        if specials:
            pool = np.array([0.0, -0.0, 1e-45, -1e-45, 1.1754942e-38, 3.4028235e38,
                             -3.4028235e38, np.inf, -np.inf], dtype=np.float32)
            m = rng.random(n) < 0.2
            x[m] = rng.choice(pool, size=m.sum())
        return x
    bits = rng.integers(0, 1 << 16, size=n, dtype=np.int64).astype(np.uint16)
    if not specials:
        # drop NaN / inf patterns
        exp_mask, fld = (0x7C00, 0x7C00) if dtype == "fp16" else (0x7F80, 0x7F80)
        bits = bits[(bits & exp_mask) != fld]
    return bits


def same_bits(a, b, dtype):
    a = np.asarray(a)
    b = np.asarray(b)
    if dtype == "fp32":
        na, nb = np.isnan(a), np.isnan(b)
        return np.array_equal(na, nb) and np.array_equal(a.view(np.uint32)[~na],
                                                          b.view(np.uint32)[~nb])
    return np.array_equal(a, b)


# --------------------------------------------------------------------- closed forms
@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 16])
def test_closed_forms(dtype, n):
    """all-ones -> N; rank r filled with r -> N(N-1)/2; one-hot -> indicator.
    Catches a dropped rank, an off-by-one in the rank loop, a wrong sign."""
    count = 37
    ones = [np.full(count, value_to_storage(1, dtype)) for _ in range(n)]
    got = storage_to_float(oracle.allreduce(ones, dtype), dtype)
    assert np.all(got == n)
    ranks = [np.full(count, value_to_storage(r, dtype)) for r in range(n)]
    got = storage_to_float(oracle.allreduce(ranks, dtype), dtype)
    assert np.all(got == n * (n - 1) // 2)
    onehot = []
    for p in range(n):
        a = np.full(count, value_to_storage(0, dtype))
        a[p] = value_to_storage(1, dtype)
        onehot.append(a)
    got = storage_to_float(oracle.allreduce(onehot, dtype), dtype)
    expect = np.zeros(count)
    expect[:n] = 1
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("dtype", ALL_DTYPES)
def test_single_rank_is_identity(dtype):
    """N=1 copies the input bit for bit (no spurious rounding or flushing)."""
    rng = np.random.default_rng(7)
    x = random_raw(rng, dtype, 4096)
    out = oracle.allreduce([x], dtype)
    assert same_bits(out, x, dtype)


def test_int32_wraps():
    """int32 sums wrap modulo 2^32 (two's complement), not saturate."""
    big = np.array([2 ** 31 - 1, -2 ** 31, 5], dtype=np.int32)
    one = np.array([1, -1, -7], dtype=np.int32)
    out = oracle.allreduce([big, one], "int32")
    assert out.tolist() == [-2 ** 31, 2 ** 31 - 1, -2]


# --------------------------------------------------------------------- golden files
def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def _parse_hex(s):
    s = s.strip()
    if s in ("inf", "-inf", "nan"):
        return float(s)
    return float.fromhex(s)


def test_golden_narrowing():
    """Hand-derived RNE cases: ties to even, overflow to inf, subnormals, signed zero."""
    n = 0
    for line in _golden_lines("ieee_narrowing_cases.txt"):
        dtype, x, expect = line.split()[:3]
        v = np.float32(_parse_hex(x))
        assert float(v) == _parse_hex(x), "fixture input not a binary32 value: " + x
        got = int(oracle.from_f32(np.array([v]), dtype)[0])
        assert got == int(expect, 16), line
        n += 1
    assert n >= 30


def test_golden_rank_order_sums():
    """Fixed rank order from x_0, fp32 accumulation, one final rounding."""
    n = 0
    for line in _golden_lines("rank_order_sums.txt"):
        dtype, vals, expect = [s.strip() for s in line.split("|")[:3]]
        xs = [np.array([value_to_storage(_parse_hex(v), dtype)]) for v in vals.split(",")]
        got = storage_to_float(oracle.allreduce(xs, dtype), dtype)[0]
        e = _parse_hex(expect)
        if math.isnan(e):
            assert math.isnan(got), line
        else:
            assert got == e and math.copysign(1, got) == math.copysign(1, e), line
        n += 1
    assert n >= 20


# --------------------------------------------------------------------- conversions
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_conversion_exhaustive_round_trip(dtype):
    """All 65536 patterns: widen then narrow is the identity (NaN stays NaN)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    wide = oracle.to_f32(bits, dtype)
    back = oracle.from_f32(wide, dtype)
    nan = np.isnan(wide)
    assert np.array_equal(back[~nan], bits[~nan])
    assert np.all(np.isnan(oracle.to_f32(back[nan], dtype)))
    # widening agrees with torch's (exact) widening on every non-NaN pattern
    ref = W.from_storage(bits, dtype).to(torch.float32).numpy()
    assert np.array_equal(wide[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    # and with the brute force's field decoding
    sample = bits[::97]
    dec = np.array([brute.decode(b, dtype) for b in sample], dtype=np.float64)
    ok = ~np.isnan(dec)
    assert np.array_equal(dec[ok], oracle.to_f32(sample, dtype)[ok].astype(np.float64))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_narrowing_matches_torch(dtype):
    """RNE narrowing vs torch's float32 -> half/bfloat16 on random values, ties,
    near-overflow values and subnormals."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-40, 40, size=200000)))
    x = x.astype(np.float32)
    # exact midpoints between adjacent targets: set the highest dropped bit only
    mid = rng.integers(0, 1 << 31, size=20000, dtype=np.int64).astype(np.uint32)
    drop = 16 if dtype == "bf16" else 13
    mid = (mid & ~np.uint32((1 << drop) - 1)) | np.uint32(1 << (drop - 1))
    x = np.concatenate([x, mid.view(np.float32)])
    x = x[np.isfinite(x)]
    got = oracle.from_f32(x, dtype)
    ref = W.to_storage(torch.from_numpy(x).to(W.TORCH_DTYPES[dtype]))
    assert np.array_equal(got, ref)


def test_fp16_narrowing_matches_struct():
    """A third implementation: Python's struct 'e' (IEEE binary16, ties to even)."""
    import struct
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * np.exp2(rng.integers(-28, 17, size=20000))).astype(np.float32)
    got = oracle.from_f32(x, "fp16")
    for v, g in zip(x.tolist(), got.tolist()):
        if abs(v) >= 65520.0:
            ref = 0x7C00 | (0x8000 if v < 0 else 0)
        else:
            ref = struct.unpack("<H", struct.pack("<e", v))[0]
        assert g == ref, (v, hex(g), hex(ref))


# --------------------------------------------------------------------- brute force
@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_brute_force_bit_equal(dtype, n):
    """The pure-Python brute force and the C oracle agree bit for bit on tiny
    random inputs with specials (overflow, subnormals, signed zeros, inf)."""
    rng = np.random.default_rng(100 + n)
    m = 257
    xs = [random_raw(rng, dtype, m * 2, specials=True)[:m] for _ in range(n)]
    m = min(len(x) for x in xs)
    xs = [x[:m] for x in xs]
    got = oracle.allreduce(xs, dtype)
    ref = brute.allreduce(xs, dtype)
    for i in range(m):
        r = ref[i]
        if dtype == "int32":
            assert int(got[i]) == r
        elif dtype == "fp32":
            g = float(got[i])
            if math.isnan(r):
                assert math.isnan(g)
            else:
                assert g == r and math.copysign(1, g) == math.copysign(1, r), (i, g, r)
        else:
            g = int(got[i])
            if math.isnan(r):
                assert math.isnan(brute.decode(g, dtype))
            else:
                assert g == brute.encode(r, dtype), (i, hex(g), r)


def test_brute_force_order_sensitive_case():
    """Reordering the ranks changes a non-associative fp32 sum; the oracle
    follows rank order (catches a reversed or pairwise summation)."""
    a = [np.array([1.0], np.float32), np.array([2 ** -24], np.float32),
         np.array([2 ** -24], np.float32)]
    assert float(oracle.allreduce(a, "fp32")[0]) == 1.0
    assert float(oracle.allreduce(a[::-1], "fp32")[0]) == 1.0 + 2 ** -23
    assert brute.allreduce(a, "fp32")[0] == 1.0
    assert brute.allreduce(a[::-1], "fp32")[0] == 1.0 + 2 ** -23


# --------------------------------------------------------------------- error bounds
@pytest.mark.parametrize("n", [2, 8, 16])
def test_fp32_error_bound(n):
    """Recursive summation bound: |fl(sum) - sum| <= (N-1) u sum|x| (u = 2^-24),
    against the exact sum from Python's math.fsum (catches a wrong operand or
    a missing rank, which break the bound by orders of magnitude)."""
    rng = np.random.default_rng(n)
    m = 5000
    xs = [rng.standard_normal(m).astype(np.float32) for _ in range(n)]
    got = oracle.allreduce(xs, "fp32").astype(np.float64)
    stack = np.stack([x.astype(np.float64) for x in xs])
    exact = np.array([math.fsum(stack[:, i]) for i in range(m)])
    bound = (n - 1) * 2.0 ** -24 * np.abs(stack).sum(axis=0)
    assert np.all(np.abs(got - exact) <= bound)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_half_outputs_within_half_ulp_of_fp32_sum(dtype):
    """Outputs are the fp32 rank-order sum rounded once: within half an ulp of
    the output type of that fp32 value."""
    rng = np.random.default_rng(3)
    m, n = 4000, 8
    xs = [random_raw(rng, dtype, m * 2)[:m] for _ in range(n)]
    m = min(len(x) for x in xs)
    xs = [x[:m] for x in xs]
    wide = np.stack([oracle.to_f32(x, dtype) for x in xs]).astype(np.float32)
    acc = wide[0].copy()
    with np.errstate(over="ignore", invalid="ignore"):  # raw patterns include huge values: inf is expected
        for p in range(1, n):
            acc = (acc + wide[p]).astype(np.float32)
    got = oracle.to_f32(oracle.allreduce(xs, dtype), dtype).astype(np.float64)
    finite = np.isfinite(got) & np.isfinite(acc)
    # ulp of the output type in the binade of the larger magnitude of the two
    mag = np.maximum(np.abs(got[finite]), np.abs(acc[finite]).astype(np.float64))
    if dtype == "fp16":
        ulp = np.spacing(mag.astype(np.float16)).astype(np.float64)
    else:
        ulp = np.exp2(np.floor(np.log2(np.maximum(mag, 2.0 ** -126))) - 7)
    assert np.all(np.abs(got[finite] - acc[finite]) <= ulp / 2)


def test_integer_valued_fp32_is_exact():
    """The N=2 fp32 workload (integers in [-8, 8]) sums exactly."""
    w = W.with_count(W.C1, 10000)
    xs = [W.to_storage(t) for t in W.rank_inputs(w)]
    got = oracle.allreduce(xs, "fp32")
    exact = sum(x.astype(np.int64) for x in xs)
    assert np.array_equal(got.astype(np.int64), exact)
    assert np.all(np.abs(xs[0]) <= 8) and np.all(xs[0] == np.round(xs[0]))


# --------------------------------------------------------------------- identities
@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("n,m", [(2, 5), (3, 17), (8, 64), (8, 1)])
def test_rs_ag_identities(dtype, n, m):
    """RS shard r == slice r of AllReduce; AG == concatenation;
    AG(RS(x)) == AllReduce(x) bit for bit."""
    rng = np.random.default_rng(n * 100 + m)
    xs = [random_raw(rng, dtype, n * m * 2)[: n * m] for _ in range(n)]
    full = oracle.allreduce(xs, dtype)
    shards = [oracle.reduce_scatter(xs, dtype, r, m) for r in range(n)]
    for r in range(n):
        assert same_bits(shards[r], full[r * m:(r + 1) * m], dtype)
    ag = oracle.allgather(shards, dtype)
    assert same_bits(ag, full, dtype)
    assert same_bits(ag, np.concatenate(shards), dtype)
    # brute force of the shard definition
    ref = brute.reduce_scatter(xs, dtype, n - 1, m)
    if dtype == "int32":
        assert shards[-1].tolist() == ref


def test_allreduce_at_and_threads_agree():
    """Sampled evaluation and the threaded form give the same bits as the plain one."""
    rng = np.random.default_rng(9)
    xs = [random_raw(rng, "bf16", 100000) for _ in range(8)]
    m = min(len(x) for x in xs)
    xs = [x[:m] for x in xs]
    full = oracle.allreduce(xs, "bf16")
    idx = rng.integers(0, m, size=1000)
    assert np.array_equal(oracle.allreduce_at(xs, "bf16", idx), full[idx])
    assert np.array_equal(oracle.allreduce(xs, "bf16", nthreads=7), full)


@pytest.mark.parametrize("n,iters", [(1, 5), (2, 3), (8, 10), (5, 1)])
def test_ring_barrier_counts(n, iters):
    """Token simulation vs the closed form: each rank hears only from its
    predecessor, iters times."""
    got = oracle.ring_barrier_counts(n, iters)
    assert got.tolist() == brute.ring_barrier_counts(n, iters)
    assert got.sum() == n * iters


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.allreduce([np.zeros(3, np.float32), np.zeros(4, np.float32)], "fp32")
    with pytest.raises(ValueError):
        oracle.allreduce([np.zeros(3, np.float32)], "fp64")
    with pytest.raises(ValueError):
        oracle.reduce_scatter([np.zeros(3, np.float32)] * 2, "fp32", 1, 2)


# --------------------------------------------------------------------- fused linear + AllReduce
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_allreduce_closed_forms(dtype):
    """All-ones weights and inputs give N*kp in every row; a one-hot input
    picks one weight column per rank; a rank's zero input drops that rank."""
    n, rows, kp = 4, 16, 32
    one = value_to_storage(1, dtype)
    ws = [np.full(rows * kp, one, np.uint16) for _ in range(n)]
    xs = [np.full(kp, one, np.uint16) for _ in range(n)]
    got = storage_to_float(oracle.linear_allreduce(ws, xs, dtype, rows, kp), dtype)
    assert np.all(got == n * kp)
    rng = np.random.default_rng(1)
    ws = [np.array([value_to_storage(v, dtype) for v in rng.integers(-3, 4, size=rows * kp)],
                   np.uint16) for _ in range(n)]
    xs = []
    for p in range(n):
        x = np.full(kp, value_to_storage(0, dtype), np.uint16)
        x[p] = one  # rank p selects its column p
        xs.append(x)
    expect = sum(storage_to_float(ws[p], dtype).reshape(rows, kp)[:, p] for p in range(n))
    got = storage_to_float(oracle.linear_allreduce(ws, xs, dtype, rows, kp), dtype)
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_allreduce_rounds_once(dtype):
    """The binary64 sum is rounded once to the output type.  Hand-derived cases
    where rounding through binary32 first would land on a tie and round to
    even, but the exact sum lies just above the tie:
      bf16: 1 + 2^-8 + 2^-30 -> 1 + 2^-7 (0x3F81); via binary32 -> 1.0 (0x3F80)
      fp16: 1 + 2^-11 + 2^-14 * 2^-14 -> 1 + 2^-10 (0x3C01); via binary32 -> 1.0
    plus the same with the sign flipped, a subnormal result and an overflow."""
    if dtype == "bf16":
        w, x, want = [0x3F80, 0x3B80, 0x3080], [0x3F80, 0x3F80, 0x3F80], 0x3F81  # 1, 2^-8, 2^-30
        sub_w, sub_x, sub_want = [0x0380], [0x3A80], 0x0008       # 2^-120 * 2^-10 = 2^-130 = 8 quanta of 2^-133
        big, inf = 0x7F7F, 0x7F80                                   # largest finite, infinity
    else:
        w, x, want = [0x3C00, 0x1000, 0x0400], [0x3C00, 0x3C00, 0x0400], 0x3C01  # 1, 2^-11, 2^-14
        sub_w, sub_x, sub_want = [0x0400], [0x1400], 0x0001        # 2^-14 * 2^-10 = 2^-24
        big, inf = 0x7BFF, 0x7C00                                   # 65504, infinity

    def run(wv, xv):
        return int(oracle.linear_allreduce([np.array(wv, np.uint16)], [np.array(xv, np.uint16)], dtype,
                                           1, len(wv))[0])

    assert run(w, x) == want
    assert run([v | 0x8000 for v in w], x) == want | 0x8000
    # exact ties go to even: 1 + half a quantum -> 1; 1 + 1.5 quanta -> 1 + 2 quanta
    one = 0x3C00 if dtype == "fp16" else 0x3F80
    half_q = 0x1000 if dtype == "fp16" else 0x3B80           # 2^-11 / 2^-8
    q = 0x1400 if dtype == "fp16" else 0x3C00                # 2^-10 / 2^-7
    assert run([one, half_q], [one, one]) == one
    assert run([one, q, half_q], [one, one, one]) == one + 2
    assert run(sub_w, sub_x) == sub_want
    assert run([big, big], [0x3C00 if dtype == "fp16" else 0x3F80] * 2) == inf


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_allreduce_matches_float64_matmul(dtype):
    """Against numpy's float64 matrix product of the concatenated shards,
    rounded once to the output type by the pure-Python brute force's generic
    rounding (a library product and an independent rounding, not the oracle's
    loop)."""
    n, rows, kp = 3, 24, 40
    rng = np.random.default_rng(2)
    ws = [W.to_storage(torch.randn(rows * kp).to(W.TORCH_DTYPES[dtype])) for _ in range(n)]
    xs = [W.to_storage(torch.randn(kp).to(W.TORCH_DTYPES[dtype])) for _ in range(n)]
    a = np.concatenate([storage_to_float(w, dtype).reshape(rows, kp) for w in ws], axis=1)
    x = np.concatenate([storage_to_float(v, dtype) for v in xs])
    ref = np.array([brute.encode(brute.round_ieee(float(v), *brute.FORMATS[dtype]), dtype) for v in a @ x],
                   np.uint16)
    got = oracle.linear_allreduce(ws, xs, dtype, rows, kp)
    # the fp64 sums of a float64 matmul may differ from the oracle's loop in the
    # last bits of binary64; after rounding to 16 bits they agree except at
    # ties, which random normal data does not produce
    assert np.array_equal(got, ref)
    del rng


# --------------------------------------------------------------------- linear layer, many tokens
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_tokens_each_token_is_the_single_token_layer(dtype):
    """Token t of the batched layer is the one-token layer applied to token t's
    slice of every rank's input, and lands at row t of the output (checks the
    token offsets of the inputs and of the output)."""
    n, tokens, rows, kp = 3, 5, 12, 24
    rng = np.random.default_rng(11)
    ws = [_small_ints(rng, dtype, -3, 3, rows * kp) for _ in range(n)]
    xs = [_small_ints(rng, dtype, -2, 2, tokens * kp) for _ in range(n)]
    got = oracle.linear_allreduce_tokens(ws, xs, dtype, tokens, rows, kp).reshape(tokens, rows)
    for t in range(tokens):
        one = oracle.linear_allreduce(ws, [x[t * kp:(t + 1) * kp] for x in xs], dtype, rows, kp)
        assert np.array_equal(got[t], one), t
    # the tokens differ, so a mix-up of rows would show
    assert len({tuple(r) for r in got}) == tokens


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_tokens_closed_forms(dtype):
    """All-ones weights with token t's inputs all equal to t+1 give N*kp*(t+1)
    in every row of token t; a rank whose inputs are all zero drops out."""
    n, tokens, rows, kp = 4, 6, 8, 16
    one = value_to_storage(1, dtype)
    ws = [np.full(rows * kp, one, np.uint16) for _ in range(n)]
    xs = [np.concatenate([np.full(kp, value_to_storage(t + 1, dtype), np.uint16) for t in range(tokens)])
          for _ in range(n)]
    got = storage_to_float(oracle.linear_allreduce_tokens(ws, xs, dtype, tokens, rows, kp), dtype)
    assert np.array_equal(got.reshape(tokens, rows), np.repeat(np.arange(1, tokens + 1)[:, None] * n * kp, rows, 1))
    xs[2] = np.full(tokens * kp, value_to_storage(0, dtype), np.uint16)
    got = storage_to_float(oracle.linear_allreduce_tokens(ws, xs, dtype, tokens, rows, kp), dtype)
    assert np.array_equal(got.reshape(tokens, rows),
                          np.repeat(np.arange(1, tokens + 1)[:, None] * (n - 1) * kp, rows, 1))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_tokens_matches_float64_matmul(dtype):
    """Against numpy's float64 matrix product X_cat @ W_cat^T of the
    concatenated shards, rounded once by the brute force's generic rounding."""
    n, tokens, rows, kp = 3, 7, 20, 32
    ws = [W.to_storage(torch.randn(rows * kp).to(W.TORCH_DTYPES[dtype])) for _ in range(n)]
    xs = [W.to_storage(torch.randn(tokens * kp).to(W.TORCH_DTYPES[dtype])) for _ in range(n)]
    a = np.concatenate([storage_to_float(w, dtype).reshape(rows, kp) for w in ws], axis=1)
    x = np.concatenate([storage_to_float(v, dtype).reshape(tokens, kp) for v in xs], axis=1)
    prod = x @ a.T  # tokens x rows
    ref = np.array([brute.encode(brute.round_ieee(float(v), *brute.FORMATS[dtype]), dtype) for v in prod.ravel()],
                   np.uint16)
    got = oracle.linear_allreduce_tokens(ws, xs, dtype, tokens, rows, kp)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_tokens_residual_reduces_to_its_parts(dtype):
    """The batched layer with residuals: zero weights give each rank its own
    residual; a zero residual gives the batched layer; every token of rank q
    equals the pinned one-token residual layer on that token's slices."""
    n, tokens, rows, kp = 3, 4, 16, 8
    rng = np.random.default_rng(23)
    ws = [_small_ints(rng, dtype, -3, 3, rows * kp) for _ in range(n)]
    xs = [_small_ints(rng, dtype, -2, 2, tokens * kp) for _ in range(n)]
    res = [_small_ints(rng, dtype, -50, 50, tokens * rows) for _ in range(n)]
    zw = [np.full(rows * kp, value_to_storage(0, dtype), np.uint16) for _ in range(n)]
    for q, y in enumerate(oracle.linear_allreduce_tokens_residual(zw, xs, res, dtype, tokens, rows, kp)):
        assert np.array_equal(storage_to_float(y, dtype), storage_to_float(res[q], dtype)), q
    zres = [np.full(tokens * rows, value_to_storage(0, dtype), np.uint16) for _ in range(n)]
    plain = oracle.linear_allreduce_tokens(ws, xs, dtype, tokens, rows, kp)
    for y in oracle.linear_allreduce_tokens_residual(ws, xs, zres, dtype, tokens, rows, kp):
        assert np.array_equal(y, plain)
    ys = oracle.linear_allreduce_tokens_residual(ws, xs, res, dtype, tokens, rows, kp)
    for t in range(tokens):
        one = oracle.linear_allreduce_residual(ws, [x[t * kp:(t + 1) * kp] for x in xs],
                                               [r[t * rows:(t + 1) * rows] for r in res], dtype, rows, kp)
        for q in range(n):
            assert np.array_equal(ys[q][t * rows:(t + 1) * rows], one[q]), (t, q)


# --------------------------------------------------------------------- linear layer + residual
def _small_ints(rng, dtype, lo, hi, size):
    return np.array([value_to_storage(int(v), dtype) for v in rng.integers(lo, hi + 1, size=size)], np.uint16)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_residual_closed_forms(dtype):
    """Zero weights leave each rank its own residual; a zero residual gives the
    layer without one; on small-integer data output q minus output 0 is
    residual q minus residual 0; (+0) + (-0) is +0."""
    n, rows, kp = 4, 16, 32
    rng = np.random.default_rng(11)
    zero = value_to_storage(0, dtype)
    ws0 = [np.full(rows * kp, zero, np.uint16) for _ in range(n)]
    xs = [_small_ints(rng, dtype, -3, 3, kp) for _ in range(n)]
    res = [_small_ints(rng, dtype, -50, 50, rows) for _ in range(n)]
    for q, y in enumerate(oracle.linear_allreduce_residual(ws0, xs, res, dtype, rows, kp)):
        assert np.array_equal(storage_to_float(y, dtype), storage_to_float(res[q], dtype))
    ws = [_small_ints(rng, dtype, -3, 3, rows * kp) for _ in range(n)]
    zres = [np.full(rows, zero, np.uint16) for _ in range(n)]
    plain = oracle.linear_allreduce(ws, xs, dtype, rows, kp)
    for y in oracle.linear_allreduce_residual(ws, xs, zres, dtype, rows, kp):
        assert np.array_equal(y, plain)
    ys = oracle.linear_allreduce_residual(ws, xs, res, dtype, rows, kp)
    base = storage_to_float(plain, dtype)
    for q in range(n):
        assert np.array_equal(storage_to_float(ys[q], dtype), base + storage_to_float(res[q], dtype))
    negz = [np.full(rows, 0x8000, np.uint16) for _ in range(n)]
    for y in oracle.linear_allreduce_residual(ws0, xs, negz, dtype, rows, kp):
        assert np.all(y == 0)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_residual_rounds_once(dtype):
    """The residual joins the exact sum before the one rounding.  Hand cases
    where rounding the layer first would leave an exact tie (to even, 1.0):
      bf16: layer 1 + 2^-30, residual 2^-8 -> 1 + 2^-7 (0x3F81)
      fp16: layer 1 + 2^-24, residual 2^-11 -> 1 + 2^-10 (0x3C01)"""
    if dtype == "bf16":
        w, x, r, want = [0x3F80, 0x3080], [0x3F80, 0x3F80], 0x3B80, 0x3F81   # 1, 2^-30; 2^-8
    else:
        w, x, r, want = [0x3C00, 0x0C00], [0x3C00, 0x0C00], 0x1000, 0x3C01   # 1, 2^-12 * 2^-12; 2^-11
    ys = oracle.linear_allreduce_residual([np.array(w, np.uint16)], [np.array(x, np.uint16)],
                                          [np.array([r], np.uint16)], dtype, 1, len(w))
    assert int(ys[0][0]) == want
    ys = oracle.linear_allreduce_residual([np.array([v | 0x8000 for v in w], np.uint16)], [np.array(x, np.uint16)],
                                          [np.array([r | 0x8000], np.uint16)], dtype, 1, len(w))
    assert int(ys[0][0]) == want | 0x8000


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_residual_matches_float64_matmul(dtype):
    """Against numpy's float64 product of the concatenated shards plus each
    rank's residual, rounded once by the brute force's generic rounding."""
    n, rows, kp = 3, 24, 40
    ws = [W.to_storage(torch.randn(rows * kp).to(W.TORCH_DTYPES[dtype])) for _ in range(n)]
    xs = [W.to_storage(torch.randn(kp).to(W.TORCH_DTYPES[dtype])) for _ in range(n)]
    res = [W.to_storage(torch.randn(rows).to(W.TORCH_DTYPES[dtype])) for _ in range(n)]
    a = np.concatenate([storage_to_float(w, dtype).reshape(rows, kp) for w in ws], axis=1)
    x = np.concatenate([storage_to_float(v, dtype) for v in xs])
    layer = a @ x
    ys = oracle.linear_allreduce_residual(ws, xs, res, dtype, rows, kp)
    for q in range(n):
        exact = layer + storage_to_float(res[q], dtype).astype(np.float64)
        ref = np.array([brute.encode(brute.round_ieee(float(v), *brute.FORMATS[dtype]), dtype) for v in exact],
                       np.uint16)
        assert np.array_equal(ys[q], ref), q


# --------------------------------------------------------------------- MAX / MIN
def test_golden_max_min():
    """Hand-derived MAX / MIN cases (tests/golden/max_min_cases.txt, IEEE 754-2019
    maximum / minimum): signed zeros both ways, NaN in any position and at one
    rank (canonical quiet NaN), infinities against the largest finite values,
    subnormals, several ranks, signed int32."""
    n = 0
    for line in _golden_lines("max_min_cases.txt"):
        dtype, op, vals, want = line.split()[:4]
        bits = [int(v, 16) for v in vals.split(",")]
        if dtype in ("fp32", "int32"):
            raw = [np.array([b], np.uint32) for b in bits]
            xs = [r.view(np.float32) if dtype == "fp32" else r.view(np.int32) for r in raw]
            got = int(np.asarray(oracle.allreduce_op(xs, dtype, op)).view(np.uint32)[0])
        else:
            xs = [np.array([b], np.uint16) for b in bits]
            got = int(np.asarray(oracle.allreduce_op(xs, dtype, op))[0])
        assert got == int(want, 16), line
        n += 1
    assert n >= 30


@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("n", [1, 2, 3, 8, 16])
def test_max_min_closed_forms(dtype, n):
    """Rank r filled with r: max N-1, min 0; rank r filled with -r: max 0,
    min -(N-1); one rank is the identity."""
    m = 37
    up = [np.full(m, value_to_storage(r, dtype)) for r in range(n)]
    down = [np.full(m, value_to_storage(-r, dtype)) for r in range(n)]
    assert np.all(storage_to_float(oracle.allreduce_op(up, dtype, "max"), dtype) == n - 1)
    assert np.all(storage_to_float(oracle.allreduce_op(up, dtype, "min"), dtype) == 0)
    assert np.all(storage_to_float(oracle.allreduce_op(down, dtype, "max"), dtype) == 0)
    assert np.all(storage_to_float(oracle.allreduce_op(down, dtype, "min"), dtype) == -(n - 1))


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_max_min_ieee_special_cases(dtype):
    """Hand cases of the IEEE 754-2019 maximum / minimum: a NaN operand gives
    NaN in either position; max(-0, +0) = +0 and min = -0 in both orders;
    infinities order; a subnormal is above zero."""
    nan, inf = float("nan"), float("inf")
    tiny = {"fp32": 1e-45, "fp16": 2.0 ** -24, "bf16": 2.0 ** -133}[dtype]
    cases = [((-0.0, 0.0), 0.0, -0.0), ((0.0, -0.0), 0.0, -0.0), ((nan, 1.0), nan, nan),
             ((1.0, nan), nan, nan), ((-inf, 3.0), 3.0, -inf), ((inf, -inf), inf, -inf),
             ((tiny, 0.0), tiny, 0.0), ((-2.0, -0.0, 5.0), 5.0, -2.0)]

    def bits(v):
        s = value_to_storage(v, dtype)
        return int(np.asarray(s).view(np.uint32 if dtype == "fp32" else np.uint16))

    for vals, want_max, want_min in cases:
        xs = [np.array([value_to_storage(v, dtype)]) for v in vals]
        for op, want in (("max", want_max), ("min", want_min)):
            got = oracle.allreduce_op(xs, dtype, op)
            g = float(storage_to_float(got, dtype)[0])
            if math.isnan(want):
                assert math.isnan(g), (vals, op)
            else:
                gb = int(np.asarray(got).view(np.uint32 if dtype == "fp32" else np.uint16)[0])
                assert gb == bits(want), (vals, op, hex(gb))


@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("op", ["max", "min"])
@pytest.mark.parametrize("n", [1, 2, 5, 8])
def test_max_min_brute_force_bit_equal(dtype, op, n):
    """The pure-Python brute force and the C oracle agree bit for bit on random
    raw patterns with NaN, infinities, subnormals and signed zeros."""
    rng = np.random.default_rng(300 + n)
    m = 301
    xs = [random_raw(rng, dtype, m * 2, specials=True)[:m] for _ in range(n)]
    m = min(len(x) for x in xs)
    xs = [x[:m] for x in xs]
    if dtype == "fp32":
        for x in xs:
            x[rng.random(m) < 0.03] = np.nan
    got = oracle.allreduce_op(xs, dtype, op)
    ref = brute.allreduce_op(xs, dtype, op)
    for i in range(m):
        r = ref[i]
        if dtype == "int32":
            assert int(got[i]) == r
        elif dtype == "fp32":
            g = float(got[i])
            if math.isnan(r):
                assert math.isnan(g)
            else:
                assert g == r and math.copysign(1, g) == math.copysign(1, r), (i, g, r)
        else:
            g = int(got[i])
            if math.isnan(r):
                assert math.isnan(brute.decode(g, dtype))
            else:
                assert g == brute.encode(r, dtype), (i, hex(g), r)


@pytest.mark.parametrize("dtype", ALL_DTYPES)
def test_max_min_match_numpy_on_finite_data(dtype):
    """Against numpy's maximum / minimum reductions (a library routine) on
    finite data, compared by value."""
    rng = np.random.default_rng(9)
    m, n = 2000, 8
    xs = [random_raw(rng, dtype, m * 2)[:m] for _ in range(n)]
    m = min(len(x) for x in xs)
    xs = [x[:m] for x in xs]
    stack = np.stack([storage_to_float(x, dtype) for x in xs])
    assert np.array_equal(storage_to_float(oracle.allreduce_op(xs, dtype, "max"), dtype), stack.max(axis=0))
    assert np.array_equal(storage_to_float(oracle.allreduce_op(xs, dtype, "min"), dtype), stack.min(axis=0))


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("n", [1, 2, 3])
def test_max_min_nan_is_canonical(dtype, n):
    """A NaN in any rank -- signalling, negative or with a payload -- gives
    the canonical quiet NaN bits, for one rank as for several."""
    canon = {"fp32": 0x7fc00000, "fp16": 0x7e00, "bf16": 0x7fc0}[dtype]
    nans = {"fp32": [0xffc00001, 0x7f800001, 0xff812345], "fp16": [0xfe01, 0x7c01, 0xfd55],
            "bf16": [0xffc1, 0x7f81, 0xff95]}[dtype]
    store = np.uint32 if dtype == "fp32" else np.uint16
    for bits in nans:
        for where in range(n):
            cols = [np.array([0x3c00 if dtype == "fp16" else (0x3f80 if dtype == "bf16" else 0x3f800000)],
                             dtype=store) for _ in range(n)]
            cols[where] = np.array([bits], dtype=store)
            xs = [c.view(np.float32) if dtype == "fp32" else c for c in cols]
            for op in ("max", "min"):
                got = oracle.allreduce_op(xs, dtype, op)
                assert int(np.asarray(got).view(store)[0]) == canon, (hex(bits), where, op)
