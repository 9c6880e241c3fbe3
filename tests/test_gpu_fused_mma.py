"""Row-parallel linear layer over a batch of tokens, fused with the AllReduce
on the tensor cores, against the oracle.

Small-integer data make every fp32 partial sum exact, so the kernel must match
the oracle bit for bit whatever order the tensor cores accumulate in.  Random
data are held to the bound of an fp32 sum of K = N*kp products (exact in
fp32) plus the KS split partials, with a unit roundoff of 2^-23 per add (so a
truncating adder is covered too), before the one rounding to the output type:
  |y - y_oracle| <= gamma_{K + KS} * sum|w x| + ulp_out,  gamma_m = m u / (1 - m u).
"""
import numpy as np
import pytest
import torch

import oracle
from driven_collective_communication_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TD = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module")
def dcc():
    from driven_collective_communication_gb300 import build
    build.build()
    from driven_collective_communication_gb300 import dcc as mod
    torch.cuda.set_device(0)
    return mod


def run(dcc, ws, xs, tokens, rows, kp, dtype, fill=float("nan")):
    n = len(ws)
    dw = [w.cuda() for w in ws]
    dx = [x.cuda() for x in xs]
    dy = [torch.full((tokens * rows,), fill, dtype=TD[dtype], device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", dw)
        for r in range(n):
            comm.register(r, "input", dx[r])
        comm.register_all("output", dy)
        dcc.dcc_linear_allreduce_tokens(comm.handle, dw, dx, dy, tokens, rows, kp, dtype)
        assert comm.check() == dcc.DCC_OK
    for r in range(1, n):
        assert torch.equal(dy[r].view(torch.int16), dy[0].view(torch.int16)), r
    return W.to_storage(dy[0])


def small_ints(g, size, dtype, lo=-3, hi=3):
    return torch.randint(lo, hi + 1, (size,), generator=g).to(TD[dtype])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("n,tokens,rows,kp", [
    (1, 1, 128, 64), (2, 16, 256, 64), (8, 1, 1024, 128), (8, 17, 1024, 192), (3, 100, 136, 256),
    (8, 256, 512, 64), (16, 64, 512, 64), (5, 255, 264, 320), (8, 33, 8192, 64), (4, 128, 128, 1024),
    (16, 256, 8, 64), (2, 1, 8, 64), (1, 255, 16, 64),
    (8, 5, 256, 72), (3, 17, 136, 200), (2, 1, 64, 8), (4, 130, 264, 1000), (8, 64, 1024, 1016)])
def test_tokens_integer_data_bit_exact(dcc, dtype, n, tokens, rows, kp):
    """Ragged token counts (padded to a multiple of 16 inside), a partial last
    row tile (136, 264 rows), tiles of 8 and 16 rows, 1..16 ranks, K splits
    from 1 to 8 (fewer where the epilogue's inbox would not fit), and kp not a
    multiple of 64 (each rank's last 64-column block partial: 8, 72, 200,
    1000, 1016)."""
    g = torch.Generator().manual_seed(n * 7919 + tokens * 31 + kp)
    ws = [small_ints(g, rows * kp, dtype) for _ in range(n)]
    xs = [small_ints(g, tokens * kp, dtype, -2, 2) for _ in range(n)]
    got = run(dcc, ws, xs, tokens, rows, kp, dtype)
    expect = oracle.linear_allreduce_tokens([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                            dtype, tokens, rows, kp)
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("form", ["pair", "one", "two"])
@pytest.mark.parametrize("n,tokens,rows,kp", [
    (1, 1, 136, 64), (2, 17, 264, 128), (8, 256, 1032, 64), (3, 200, 200, 192), (8, 64, 8192, 64),
    (16, 130, 520, 64), (8, 1, 8192, 128), (4, 33, 1000, 64), (2, 16, 520, 64), (8, 96, 1032, 136)])
def test_tokens_every_form_bit_exact(dcc, monkeypatch, form, n, tokens, rows, kp):
    """Every form of the kernel (128-thread CTAs two per SM with one
    accumulator; 256-thread CTAs one per SM with one accumulator of up to 128
    rows, or two sharing the token tile, up to 256 rows -- one where the rows,
    tensor memory or the epilogue's room do not allow two) on the same shapes,
    whatever the token count would pick: partial last accumulators (136, 200,
    264 rows), residuals."""
    monkeypatch.setenv("DCC_MMA_FORM", form)
    g = torch.Generator().manual_seed(n * 17 + tokens + rows)
    ws = [small_ints(g, rows * kp, "bf16") for _ in range(n)]
    xs = [small_ints(g, tokens * kp, "bf16", -2, 2) for _ in range(n)]
    got = run(dcc, ws, xs, tokens, rows, kp, "bf16")
    expect = oracle.linear_allreduce_tokens([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                            "bf16", tokens, rows, kp)
    assert np.array_equal(got, expect)
    res = [small_ints(g, tokens * rows, "bf16", -50, 50) for _ in range(n)]
    got = run_residual(dcc, ws, xs, res, tokens, rows, kp, "bf16", inplace=True)
    expect = oracle.linear_allreduce_tokens_residual([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                                     [W.to_storage(r) for r in res], "bf16", tokens, rows, kp)
    for q in range(n):
        assert np.array_equal(got[q], expect[q]), q


def test_tokens_random_shapes_bit_exact(dcc):
    """Forty seeded random mixes of rank count, tokens, rows, kp and dtype on
    small-integer data: exact against the oracle."""
    rng = np.random.default_rng(2026)
    for case in range(40):
        n = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
        tokens = int(rng.integers(1, 257))
        rows = 8 * int(rng.integers(1, 80))
        kp = 64 * int(rng.integers(1, 9))
        dtype = str(rng.choice(["bf16", "fp16"]))
        g = torch.Generator().manual_seed(5000 + case)
        ws = [small_ints(g, rows * kp, dtype) for _ in range(n)]
        xs = [small_ints(g, tokens * kp, dtype, -2, 2) for _ in range(n)]
        got = run(dcc, ws, xs, tokens, rows, kp, dtype)
        expect = oracle.linear_allreduce_tokens([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                                dtype, tokens, rows, kp)
        assert np.array_equal(got, expect), (case, n, tokens, rows, kp, dtype)


def ulp_out(v, dtype):
    big = np.maximum(np.abs(v), 2.0 ** (-126 if dtype == "bf16" else -14))
    return np.exp2(np.floor(np.log2(big)) - (7 if dtype == "bf16" else 10))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("n,tokens,rows,kp", [(8, 64, 1024, 1024), (8, 256, 256, 512), (3, 5, 264, 2048)])
def test_tokens_random_data_within_bound(dcc, dtype, n, tokens, rows, kp):
    g = torch.Generator().manual_seed(17 + n + kp + tokens)
    ws = [(torch.randn(rows * kp, generator=g) * 0.05).to(TD[dtype]) for _ in range(n)]
    xs = [torch.randn(tokens * kp, generator=g).to(TD[dtype]) for _ in range(n)]
    got = run(dcc, ws, xs, tokens, rows, kp, dtype)
    expect = oracle.linear_allreduce_tokens([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                            dtype, tokens, rows, kp)
    gf = W.from_storage(got, dtype).double().numpy()
    ef = W.from_storage(expect, dtype).double().numpy()
    s = sum(np.abs(x.double().numpy().reshape(tokens, kp)) @ np.abs(w.double().numpy().reshape(rows, kp)).T
            for w, x in zip(ws, xs)).ravel()
    m = n * kp + 8  # products plus at most 8 split partials
    u = 2.0 ** -23
    gamma = m * u / (1 - m * u)
    bound = gamma * s + ulp_out(np.maximum(np.abs(gf), np.abs(ef)), dtype)
    assert np.all(np.abs(gf - ef) <= bound), float(np.max(np.abs(gf - ef) / bound))
    assert np.mean(got == expect) > 0.9


def test_tokens_full_size_sampled_rows(dcc):
    """8 ranks x 8192 rows x kp 1024, 256 tokens (the bench's largest batch),
    integer data: 1024 rows spread over the matrix (every row tile touched,
    the first and last rows included) against the oracle, every token."""
    n, tokens, rows, kp, dtype = 8, 256, 8192, 1024, "bf16"
    g = torch.Generator().manual_seed(99)
    ws = [small_ints(g, rows * kp, dtype) for _ in range(n)]
    xs = [small_ints(g, tokens * kp, dtype, -2, 2) for _ in range(n)]
    got = run(dcc, ws, xs, tokens, rows, kp, dtype).reshape(tokens, rows)
    pick = np.unique(np.concatenate([np.arange(0, rows, 8), [rows - 1]]))[:1025]
    wsel = [W.to_storage(w).reshape(rows, kp)[pick].ravel() for w in ws]
    expect = oracle.linear_allreduce_tokens(wsel, [W.to_storage(x) for x in xs], dtype, tokens, len(pick),
                                            kp).reshape(tokens, len(pick))
    assert np.array_equal(got[:, pick], expect)


def test_tokens_argument_errors(dcc):
    n, tokens, rows, kp = 2, 4, 64, 64
    w = [torch.zeros(rows * kp, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    x = [torch.zeros(tokens * kp, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    y = [torch.zeros(tokens * rows, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", w)
        comm.register_all("input", x)
        comm.register_all("output", y)
        h = comm.handle

        def code(*args):
            try:
                dcc.dcc_linear_allreduce_tokens(h, *args)
                return dcc.DCC_OK
            except dcc.DccError as e:
                return e.code
        assert code(w, x, y, tokens, rows, kp, "bf16") == dcc.DCC_OK
        assert code(w, x, y, 0, rows, kp, "bf16") == dcc.DCC_OK          # nothing to do
        assert code(w, x, y, 257, rows, kp, "bf16") == dcc.DCC_ERR_UNSUPPORTED
        assert code(w, x, y, tokens, rows, 12, "bf16") == dcc.DCC_ERR_UNSUPPORTED  # kp % 8
        assert code(w, x, y, tokens, 60, kp, "bf16") == dcc.DCC_ERR_UNSUPPORTED   # rows % 8
        assert code(w, x, y, tokens, rows, kp, "fp32") == dcc.DCC_ERR_UNSUPPORTED
        assert code(w, x, y, tokens, rows * 2, kp, "bf16") == dcc.DCC_ERR_NOT_REGISTERED
        bad = [t[1:] for t in y]
        assert code(w, x, bad, tokens, rows - 8, kp, "bf16") == dcc.DCC_ERR_MISALIGNED
        assert code(w, x, [y[0], y[0]], tokens, rows, kp, "bf16") == dcc.DCC_ERR_NOT_REGISTERED  # not rank 1's
        comm.register(1, "output", y[0])
        assert code(w, x, [y[0], y[0]], tokens, rows, kp, "bf16") == dcc.DCC_ERR_INVALID_ARG  # outputs overlap
        assert code(w, x, [x[0], y[1]], tokens, rows, kp, "bf16") == dcc.DCC_ERR_INVALID_ARG  # output is an input
        assert comm.check() == dcc.DCC_OK


def run_residual(dcc, ws, xs, res, tokens, rows, kp, dtype, inplace=False):
    n = len(ws)
    dw = [w.cuda() for w in ws]
    dx = [x.cuda() for x in xs]
    dr = [r.cuda() for r in res]
    dy = dr if inplace else [torch.full((tokens * rows,), float("nan"), dtype=TD[dtype], device="cuda")
                             for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", dw)
        for r in range(n):
            comm.register(r, "input", dx[r])
        comm.register_all("output", dy)
        if not inplace:
            comm.register_all("input", dr)
        dcc.dcc_linear_allreduce_tokens_residual(comm.handle, dw, dx, dr, dy, tokens, rows, kp, dtype)
        assert comm.check() == dcc.DCC_OK
    return [W.to_storage(y) for y in dy]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("n,tokens,rows,kp,inplace", [
    (1, 1, 128, 64, False), (2, 16, 256, 64, True), (8, 17, 1024, 192, False), (3, 100, 136, 256, True),
    (8, 256, 512, 64, False), (16, 64, 512, 64, True), (5, 255, 264, 320, False), (8, 33, 8192, 64, True)])
def test_tokens_residual_integer_data_bit_exact(dcc, dtype, n, tokens, rows, kp, inplace):
    """Each rank's output is the batched layer plus its own residual, exact on
    small-integer data; in place the residual buffer is the output."""
    g = torch.Generator().manual_seed(n * 131 + tokens * 7 + kp + int(inplace))
    ws = [small_ints(g, rows * kp, dtype) for _ in range(n)]
    xs = [small_ints(g, tokens * kp, dtype, -2, 2) for _ in range(n)]
    res = [small_ints(g, tokens * rows, dtype, -100, 100) for _ in range(n)]
    got = run_residual(dcc, ws, xs, res, tokens, rows, kp, dtype, inplace)
    expect = oracle.linear_allreduce_tokens_residual([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                                     [W.to_storage(r) for r in res], dtype, tokens, rows, kp)
    for q in range(n):
        assert np.array_equal(got[q], expect[q]), q


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_tokens_residual_random_data_within_bound(dcc, dtype):
    n, tokens, rows, kp = 8, 64, 1024, 1024
    g = torch.Generator().manual_seed(404)
    ws = [(torch.randn(rows * kp, generator=g) * 0.05).to(TD[dtype]) for _ in range(n)]
    xs = [torch.randn(tokens * kp, generator=g).to(TD[dtype]) for _ in range(n)]
    res = [torch.randn(tokens * rows, generator=g).to(TD[dtype]) for _ in range(n)]
    got = run_residual(dcc, ws, xs, res, tokens, rows, kp, dtype)
    expect = oracle.linear_allreduce_tokens_residual([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                                     [W.to_storage(r) for r in res], dtype, tokens, rows, kp)
    s = sum(np.abs(x.double().numpy().reshape(tokens, kp)) @ np.abs(w.double().numpy().reshape(rows, kp)).T
            for w, x in zip(ws, xs)).ravel()
    m = n * kp + 8 + 1  # products, at most 8 split partials, the residual
    u = 2.0 ** -23
    gamma = m * u / (1 - m * u)
    for q in range(n):
        gf = W.from_storage(got[q], dtype).double().numpy()
        ef = W.from_storage(expect[q], dtype).double().numpy()
        rq = np.abs(res[q].double().numpy())
        bound = gamma * (s + rq) + ulp_out(np.maximum(np.abs(gf), np.abs(ef)), dtype)
        assert np.all(np.abs(gf - ef) <= bound), (q, float(np.max(np.abs(gf - ef) / bound)))
        assert np.mean(got[q] == expect[q]) > 0.9


def test_tokens_residual_argument_errors(dcc):
    n, tokens, rows, kp = 2, 4, 64, 64
    z = lambda size: torch.zeros(size, dtype=torch.bfloat16, device="cuda")
    w = [z(rows * kp) for _ in range(n)]
    x = [z(tokens * kp) for _ in range(n)]
    y = [z(tokens * rows) for _ in range(n)]
    res = [z(tokens * rows + 8) for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", w)
        comm.register_all("input", x)
        comm.register_all("output", y)
        h = comm.handle

        def code(*args):
            try:
                dcc.dcc_linear_allreduce_tokens_residual(h, *args)
                return dcc.DCC_OK
            except dcc.DccError as e:
                return e.code
        assert dcc.raw_call("dcc_linear_allreduce_tokens_residual", h, dcc._ptrs(w), dcc._ptrs(x), None,
                            dcc._ptrs(y), tokens, rows, kp, dcc._dtype("bf16"), None) == dcc.DCC_ERR_INVALID_ARG
        assert code(w, x, res, y, tokens, rows, kp, "bf16") == dcc.DCC_ERR_NOT_REGISTERED
        comm.register_all("input", res)
        assert code(w, x, res, y, tokens, rows, kp, "bf16") == dcc.DCC_OK
        assert code(w, x, y, y, tokens, rows, kp, "bf16") == dcc.DCC_OK                      # in place
        assert code(w, x, [r[1:] for r in res], y, tokens, rows, kp, "bf16") == dcc.DCC_ERR_MISALIGNED
        assert code(w, x, [y[1], y[0]], y, tokens, rows, kp, "bf16") == dcc.DCC_ERR_NOT_REGISTERED
        comm.register(0, "output", y[1])
        comm.register(1, "output", y[0])
        assert code(w, x, [y[1], y[0]], y, tokens, rows, kp, "bf16") == dcc.DCC_ERR_INVALID_ARG  # another's output
        assert comm.check() == dcc.DCC_OK


@pytest.mark.parametrize("rows,tokens,threads,macc,min_ks", [
    (8192, 1, 128, 1, 4), (8192, 96, 128, 1, 4), (8192, 97, 256, 1, 1), (8192, 256, 256, 1, 1),
    (4096, 96, 256, 1, 4), (28672, 1, 128, 1, 1), (28672, 256, 256, 2, 1)])
def test_tokens_form_by_shape(dcc, monkeypatch, capfd, rows, tokens, threads, macc, min_ks):
    """The launch the library picks for 8 ranks x kp 1024: at 8192 rows (the
    decode shape) up to 96 tokens the pair form (128-thread CTAs, two per SM)
    with a K split of at least 4, above it 256-thread CTAs with one
    accumulator; at 4096 rows, where both forms fit a 4-way split in one
    wave, the 256-thread form; at 28672 rows x 256 tokens, where only two
    accumulators per CTA fit the tiles in one wave, that form.  Read from the
    library's launch log."""
    monkeypatch.setenv("DCC_LOG", "1")
    n, kp = 8, 1024
    w = [torch.zeros(rows * kp, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    x = [torch.zeros(tokens * kp, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    y = [torch.empty(tokens * rows, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", w)
        comm.register_all("input", x)
        comm.register_all("output", y)
        capfd.readouterr()
        dcc.dcc_linear_allreduce_tokens(comm.handle, w, x, y, tokens, rows, kp, "bf16")
        torch.cuda.synchronize()
        err = capfd.readouterr().err
        assert comm.check() == dcc.DCC_OK
    line = [l for l in err.splitlines() if "dcc_linear_allreduce_tokens:" in l][-1]
    fields = dict(f.split("=") for f in line.split() if "=" in f)
    assert int(fields["threads"]) == threads, line
    assert int(fields["macc"]) == macc, line
    assert int(fields["ks"]) >= min_ks, line
    assert int(fields["one_wave"]) == 1, line
    assert all(float(v) == 0 for v in y[0].float()[:64]), "zero weights give zero"


def test_tokens_plans_cached_across_communicators(dcc, monkeypatch):
    """Launch plans are cached per communicator and shape, and a kernel's
    shared-memory limit only ever rises: two communicators alive at once
    alternating a large token tile (more shared memory per CTA) with a small
    one on the same kernel, each call bit-exact against the oracle."""
    monkeypatch.setenv("DCC_MMA_FORM", "pair")
    n, rows, kp = 8, 1024, 128
    g = torch.Generator().manual_seed(4242)
    ws = [small_ints(g, rows * kp, "bf16") for _ in range(n)]
    dw = [w.cuda() for w in ws]
    cases = {}
    for tokens in (256, 16):
        xs = [small_ints(g, tokens * kp, "bf16", -2, 2) for _ in range(n)]
        expect = oracle.linear_allreduce_tokens([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                                "bf16", tokens, rows, kp)
        cases[tokens] = ([x.cuda() for x in xs], expect)
    with dcc.Comm(n) as big, dcc.Comm(n) as small:
        comms = {256: big, 16: small}
        outs = {t: [torch.empty(t * rows, dtype=torch.bfloat16, device="cuda") for _ in range(n)] for t in cases}
        for t, comm in comms.items():
            comm.register_all("input", dw)
            comm.register_all("input", cases[t][0])
            comm.register_all("output", outs[t])
        for tokens in (256, 16, 256, 16, 256):
            for y in outs[tokens]:
                y.fill_(float("nan"))
            rc = dcc.dcc_linear_allreduce_tokens(comms[tokens].handle, dw, cases[tokens][0], outs[tokens], tokens,
                                                 rows, kp, "bf16")
            assert rc == dcc.DCC_OK
            assert comms[tokens].check() == dcc.DCC_OK
            for r in range(n):
                assert np.array_equal(W.to_storage(outs[tokens][r]), cases[tokens][1]), (tokens, r)
