"""Row-parallel linear layer fused with the AllReduce, against the oracle.

Small-integer data make every fp32 partial sum exact, so the kernel must match
the oracle bit for bit whatever its internal order.  Random data are held to
the fp32 dot-product bound of the kernel that ran.  The thread-load and
bulk-copy kernels sum each rank's kp products with fused multiply-adds (one
rounding each) and a shuffle tree, then add the N partials, so
|acc - exact| <= gamma_{kp+N} * sum|w x| with gamma_m = m u / (1 - m u),
u = 2^-24 (round to nearest).  The tensor-core kernel accumulates the N*kp products in the tensor core's own order and then adds
its K-split partials: gamma_{N kp + KS} with u = 2^-23 (which also covers a
truncating adder), KS <= 8.  The kernel and the oracle then round once each to
the output type, which adds at most one output ulp:
  |y - y_oracle| <= gamma * sum|w x| + ulp_out.
"""
import ctypes

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


@pytest.fixture(params=["thread", "bulk", "tensor"])
def path(request, monkeypatch):
    """Every kernel of the op: thread loads (fused.cuh), bulk copies
    (fused_bulk.cuh) and the tensor-core kernel (fused_mma.cuh)."""
    monkeypatch.setenv("DCC_FUSED_KERNEL", request.param)
    return request.param


def gamma(m, u=2.0 ** -24):
    return m * u / (1 - m * u)


def dot_gamma(path, n, kp, extra=0):
    """The bound's factor for the kernel `path` runs (see the module docstring)."""
    if path == "tensor":
        return gamma(n * kp + 8 + extra, 2.0 ** -23)
    return gamma(kp + n + extra)


def run(dcc, ws, xs, rows, kp, dtype):
    n = len(ws)
    dw = [w.cuda() for w in ws]
    dx = [x.cuda() for x in xs]
    dy = [torch.full((rows,), float("nan"), dtype=TD[dtype], device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", dw)
        for r in range(n):
            comm.register(r, "input", dx[r])
        comm.register_all("output", dy)
        dcc.dcc_linear_allreduce(comm.handle, dw, dx, dy, rows, kp, dtype)
        assert comm.check() == dcc.DCC_OK
    for r in range(1, n):
        assert torch.equal(dy[r].view(torch.int16), dy[0].view(torch.int16))
    return W.to_storage(dy[0])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("n,rows,kp", [(1, 8, 8), (2, 64, 40), (8, 1032, 1032), (16, 256, 1024),
                                        (5, 136, 2056), (8, 8192, 64), (3, 24, 9000), (8, 64, 4096)])
def test_integer_data_bit_exact(dcc, path, dtype, n, rows, kp):
    g = torch.Generator().manual_seed(n * 1000 + kp)
    ws = [torch.randint(-3, 4, (rows * kp,), generator=g).to(TD[dtype]) for _ in range(n)]
    xs = [torch.randint(-3, 4, (kp,), generator=g).to(TD[dtype]) for _ in range(n)]
    got = run(dcc, ws, xs, rows, kp, dtype)
    expect = oracle.linear_allreduce([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                     dtype, rows, kp)
    assert np.array_equal(got, expect)


def test_random_shapes_bit_exact(dcc, monkeypatch):
    """Sixty seeded random mixes of rank count, rows, kp, dtype and kernel
    (thread loads / bulk copies / tensor cores) on small-integer data: exact
    against the oracle."""
    rng = np.random.default_rng(31)
    for case in range(60):
        n = int(rng.choice([1, 2, 3, 5, 8, 9, 16]))
        rows = 8 * int(rng.integers(1, 40))
        kernel = str(rng.choice(["thread", "bulk", "tensor"]))
        kp = 8 * int(rng.integers(1, 1150))
        dtype = str(rng.choice(["bf16", "fp16"]))
        monkeypatch.setenv("DCC_FUSED_KERNEL", kernel)
        g = torch.Generator().manual_seed(1000 + case)
        ws = [torch.randint(-3, 4, (rows * kp,), generator=g).to(TD[dtype]) for _ in range(n)]
        xs = [torch.randint(-3, 4, (kp,), generator=g).to(TD[dtype]) for _ in range(n)]
        got = run(dcc, ws, xs, rows, kp, dtype)
        expect = oracle.linear_allreduce([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                         dtype, rows, kp)
        assert np.array_equal(got, expect), (case, n, rows, kp, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("n,rows,kp", [(8, 8192, 1024), (8, 512, 3584), (3, 64, 4104)])
def test_random_data_within_bound(dcc, path, dtype, n, rows, kp):
    g = torch.Generator().manual_seed(7 + n + kp)
    ws = [(torch.randn(rows * kp, generator=g) * 0.05).to(TD[dtype]) for _ in range(n)]
    xs = [torch.randn(kp, generator=g).to(TD[dtype]) for _ in range(n)]
    got = run(dcc, ws, xs, rows, kp, dtype)
    expect = oracle.linear_allreduce([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                     dtype, rows, kp)
    gf = W.from_storage(got, dtype).double().numpy()
    ef = W.from_storage(expect, dtype).double().numpy()
    s = sum(np.abs(w.double().numpy().reshape(rows, kp)) @ np.abs(x.double().numpy())
            for w, x in zip(ws, xs))
    big = np.maximum(np.abs(gf), np.abs(ef))
    ulp = np.abs(np.spacing(big.astype(np.float16 if dtype == "fp16" else np.float32)).astype(np.float64))
    if dtype == "bf16":
        ulp = np.exp2(np.floor(np.log2(np.maximum(big, 2.0 ** -126))) - 7)
    bound = dot_gamma(path, n, kp) * s + ulp
    assert np.all(np.abs(gf - ef) <= bound)
    # and nearly always the same bits
    assert np.mean(got == expect) > (0.9 if path == "tensor" else 0.98)


def test_argument_errors(dcc):
    n, rows, kp = 2, 16, 16
    ws = [torch.zeros(rows * kp, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    xs = [torch.zeros(kp, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    ys = [torch.zeros(rows, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", ws)
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        h = comm.handle
        for args, code in [((rows - 1, kp, "bf16"), dcc.DCC_ERR_UNSUPPORTED),
                           ((rows, kp - 4, "bf16"), dcc.DCC_ERR_UNSUPPORTED),
                           ((rows, kp, "fp32"), dcc.DCC_ERR_UNSUPPORTED),
                           ((rows * 2, kp, "bf16"), dcc.DCC_ERR_NOT_REGISTERED)]:
            with pytest.raises(dcc.DccError) as e:
                dcc.dcc_linear_allreduce(h, ws, xs, ys, *args)
            assert e.value.code == code, args
        with pytest.raises(dcc.DccError) as e:  # output overlapping a weight
            dcc.dcc_linear_allreduce(h, ws, xs, [ws[0][:rows], ys[1]], rows, kp, "bf16")
        assert e.value.code == dcc.DCC_ERR_INVALID_ARG
        assert comm.check() == dcc.DCC_OK


# ------------------------------------------------------------------ residual epilogue
def run_residual(dcc, ws, xs, res, rows, kp, dtype, inplace):
    """dcc_linear_allreduce_residual; in place the residual buffers are the outputs.
    Returns every rank's output as raw storage."""
    n = len(ws)
    dw = [w.cuda() for w in ws]
    dx = [x.cuda() for x in xs]
    dr = [r.cuda() for r in res]
    dy = dr if inplace else [torch.full((rows,), float("nan"), dtype=TD[dtype], device="cuda") for _ in range(n)]
    with dcc.Comm(n) as comm:
        comm.register_all("input", dw)
        for r in range(n):
            comm.register(r, "input", dx[r])
        comm.register_all("output", dy)
        if not inplace:
            comm.register_all("input", dr)
        dcc.dcc_linear_allreduce_residual(comm.handle, dw, dx, dr, dy, rows, kp, dtype)
        assert comm.check() == dcc.DCC_OK
    return [W.to_storage(y) for y in dy]


def small_int_case(seed, n, rows, kp, dtype):
    g = torch.Generator().manual_seed(seed)
    ws = [torch.randint(-3, 4, (rows * kp,), generator=g).to(TD[dtype]) for _ in range(n)]
    xs = [torch.randint(-3, 4, (kp,), generator=g).to(TD[dtype]) for _ in range(n)]
    res = [torch.randint(-100, 101, (rows,), generator=g).to(TD[dtype]) for _ in range(n)]
    return ws, xs, res


def residual_expect(ws, xs, res, dtype, rows, kp):
    return oracle.linear_allreduce_residual([W.to_storage(w) for w in ws], [W.to_storage(x) for x in xs],
                                            [W.to_storage(r) for r in res], dtype, rows, kp)


@pytest.mark.parametrize("inplace", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("n,rows,kp", [(1, 8, 8), (2, 64, 40), (8, 1032, 1032), (16, 256, 1024),
                                        (3, 24, 9000), (8, 64, 4096)])
def test_residual_integer_data_bit_exact(dcc, path, dtype, n, rows, kp, inplace):
    """Each rank's own residual (they differ) joins the sum before the rounding:
    exact against the oracle on small-integer data, in and out of place."""
    ws, xs, res = small_int_case(n * 7 + kp, n, rows, kp, dtype)
    expect = residual_expect(ws, xs, res, dtype, rows, kp)
    got = run_residual(dcc, ws, xs, res, rows, kp, dtype, inplace)
    for q in range(n):
        assert np.array_equal(got[q], expect[q]), q


def test_residual_random_shapes_bit_exact(dcc, monkeypatch):
    """Thirty seeded random mixes of rank count, rows, kp, dtype, kernel and
    in / out of place with residuals, small-integer data, exact."""
    rng = np.random.default_rng(37)
    for case in range(30):
        n = int(rng.choice([1, 2, 3, 5, 8, 16]))
        rows = 8 * int(rng.integers(1, 40))
        kernel = str(rng.choice(["thread", "bulk", "tensor"]))
        kp = 8 * int(rng.integers(1, 1150))
        dtype = str(rng.choice(["bf16", "fp16"]))
        inplace = bool(rng.integers(0, 2))
        monkeypatch.setenv("DCC_FUSED_KERNEL", kernel)
        ws, xs, res = small_int_case(2000 + case, n, rows, kp, dtype)
        expect = residual_expect(ws, xs, res, dtype, rows, kp)
        got = run_residual(dcc, ws, xs, res, rows, kp, dtype, inplace)
        for q in range(n):
            assert np.array_equal(got[q], expect[q]), (case, n, rows, kp, dtype, inplace, q)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_residual_random_data_within_bound(dcc, path, dtype):
    """Random data: within the fp32 bound of the layer plus the residual term
    (one more add), |y - y_oracle| <= gamma_{m+1} (sum|w x| + |res|) + ulp with
    the kernel's m (module docstring)."""
    n, rows, kp = 8, 1024, 1024
    g = torch.Generator().manual_seed(77)
    ws = [(torch.randn(rows * kp, generator=g) * 0.05).to(TD[dtype]) for _ in range(n)]
    xs = [torch.randn(kp, generator=g).to(TD[dtype]) for _ in range(n)]
    res = [torch.randn(rows, generator=g).to(TD[dtype]) for _ in range(n)]
    expect = residual_expect(ws, xs, res, dtype, rows, kp)
    got = run_residual(dcc, ws, xs, res, rows, kp, dtype, False)
    s = sum(np.abs(w.double().numpy().reshape(rows, kp)) @ np.abs(x.double().numpy()) for w, x in zip(ws, xs))
    for q in range(n):
        gf = W.from_storage(got[q], dtype).double().numpy()
        ef = W.from_storage(expect[q], dtype).double().numpy()
        big = np.maximum(np.abs(gf), np.abs(ef))
        if dtype == "bf16":
            ulp = np.exp2(np.floor(np.log2(np.maximum(big, 2.0 ** -126))) - 7)
        else:
            ulp = np.abs(np.spacing(big.astype(np.float16)).astype(np.float64))
        bound = dot_gamma(path, n, kp, 1) * (s + np.abs(res[q].double().numpy())) + ulp
        assert np.all(np.abs(gf - ef) <= bound), q
        assert np.mean(got[q] == expect[q]) > (0.9 if path == "tensor" else 0.98)


def test_residual_argument_errors(dcc):
    """Residual overlapping another rank's output or part of its own, not
    registered, misaligned, or a NULL array: rejected, nothing launched."""
    n, rows, kp = 2, 16, 16
    ws = [torch.zeros(rows * kp, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    xs = [torch.zeros(kp, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    ys = [torch.full((rows + 64,), 5.0, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    rs = [torch.zeros(rows + 64, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    loose = torch.zeros(rows, dtype=torch.bfloat16, device="cuda")
    with dcc.Comm(n) as comm:
        comm.register_all("input", ws)
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        comm.register_all("input", rs)
        comm.register(0, "input", ys[1])  # so that the overlap check, not the window check, decides
        h = comm.handle
        y = [t[:rows] for t in ys]
        cases = [([ys[1][:rows], rs[1][:rows]], dcc.DCC_ERR_INVALID_ARG),     # rank 0's residual is rank 1's output
                 ([ys[0][8:8 + rows], rs[1][:rows]], dcc.DCC_ERR_INVALID_ARG),  # part of its own output
                 ([loose, rs[1][:rows]], dcc.DCC_ERR_NOT_REGISTERED),
                 ([rs[0][1:1 + rows], rs[1][:rows]], dcc.DCC_ERR_MISALIGNED)]
        for res, code in cases:
            with pytest.raises(dcc.DccError) as e:
                dcc.dcc_linear_allreduce_residual(h, ws, xs, res, y, rows, kp, "bf16")
            assert e.value.code == code
        P = ctypes.c_void_p * n
        rc = dcc.raw_call("dcc_linear_allreduce_residual", h, P(*[w.data_ptr() for w in ws]),
                          P(*[x.data_ptr() for x in xs]), None, P(*[t.data_ptr() for t in y]), rows, kp, 3, None)
        assert rc == dcc.DCC_ERR_INVALID_ARG
        assert comm.check() == dcc.DCC_OK
    torch.cuda.synchronize()
    for t in ys:
        assert torch.all(t == 5.0)
