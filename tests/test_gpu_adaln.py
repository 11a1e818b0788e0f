"""adaln_fwd / adaln_bwd (fused LayerNorm-Modulate, "AdaptiveLoad" §2.B)
against the fp64 oracle (GPU).

Tolerances, from the arithmetic: the kernels compute in fp32 from the bf16
inputs the oracle also sees, so y and dx differ from the oracle mainly by
their rounding to bf16 (at most 2^-9 relative); per element
|err| <= 2^-8 |ref| + 1e-3 and ||err||_2 / ||ref||_2 <= 5e-3.  dshift and
dscale stay in fp32 (sums over the tokens): ||err||_2 / ||ref||_2 <= 1e-4.
"""

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

REL_ELEM = 2.0 ** -8
ABS_ELEM = 1e-3
REL_L2_BF16 = 5e-3
REL_L2_F32 = 1e-4


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def check_bf16(name, got, ref):
    assert np.isfinite(got).all(), name
    err = np.abs(got - ref)
    bad = err > REL_ELEM * np.abs(ref) + ABS_ELEM
    assert not bad.any(), f"{name}: {bad.sum()} elements out of tolerance, worst {err.max():.3e}"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= REL_L2_BF16, f"{name}: rel L2 {rel:.3e}"


def check_f32(name, got, ref):
    assert np.isfinite(got).all(), name
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= REL_L2_F32, f"{name}: rel L2 {rel:.3e}"


def inputs(B, N, D, seed, offset=0.0, const_rows=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, N, D, generator=g) * 2.0 + offset + torch.randn(B, N, 1, generator=g)
    if const_rows:
        x[:, :const_rows] = torch.randn(B, const_rows, 1, generator=g)
    x = x.to(torch.bfloat16)
    shift = torch.randn(B, D, generator=g)
    scale = torch.randn(B, D, generator=g) * 0.3
    dy = torch.randn(B, N, D, generator=g).to(torch.bfloat16)
    return x, shift, scale, dy


def run(pvl, x, shift, scale, dy, eps):
    xc, sc, cc, dyc = x.cuda(), shift.cuda(), scale.cuda(), dy.cuda()
    y, mean, rstd = pvl.adaln_fwd(xc, sc, cc, eps, stats=True)
    dx, dshift, dscale = pvl.adaln_bwd(xc, cc, dyc, eps)
    pvl.device_error()
    return y, mean, rstd, dx, dshift, dscale


@pytest.mark.parametrize("B,N,D", [(2, 7, 8), (3, 130, 64), (2, 257, 1536), (1, 300, 3072), (2, 129, 5120),
                                   (1, 65, 8192), (1, 1, 2048), (2, 64, 5128),
                                   # more rows than CTAs: row ranges that cross batch rows
                                   (3000, 3, 1024), (5, 4001, 512), (2, 70000, 64), (3, 9001, 5120)])
def test_against_oracle(pvl, B, N, D):
    x, shift, scale, dy = inputs(B, N, D, seed=B * 1000 + N + D)
    eps = 1e-6
    y, mean, rstd, dx, dshift, dscale = run(pvl, x, shift, scale, dy, eps)
    Y, MU, R = oracle.adaln_fwd(x, shift, scale, eps)
    DX, DS, DC = oracle.adaln_bwd(x, shift, scale, dy, eps)
    check_bf16("y", to_np(y), Y)
    np.testing.assert_allclose(to_np(mean), MU, rtol=0, atol=1e-4 * (1 + np.abs(MU).max()))
    np.testing.assert_allclose(to_np(rstd), R, rtol=1e-4, atol=0)
    check_bf16("dx", to_np(dx), DX)
    check_f32("dshift", to_np(dshift), DS)
    check_f32("dscale", to_np(dscale), DC)


def test_large_offset_and_constant_rows(pvl):
    """Rows with a mean of 100 (two-pass variance) and rows that are constant
    (xh = 0: y = shift exactly, no dscale contribution)."""
    x, shift, scale, dy = inputs(2, 100, 1024, seed=5, offset=100.0, const_rows=9)
    eps = 1e-5
    y, _, _, dx, dshift, dscale = run(pvl, x, shift, scale, dy, eps)
    Y, _, _ = oracle.adaln_fwd(x, shift, scale, eps)
    DX, DS, DC = oracle.adaln_bwd(x, shift, scale, dy, eps)
    check_bf16("y", to_np(y), Y)
    const = to_np(y)[:, :9]
    exp = shift.to(torch.bfloat16).double().numpy()[:, None, :]
    np.testing.assert_array_equal(const, np.broadcast_to(exp, const.shape))
    check_bf16("dx", to_np(dx), DX)
    check_f32("dshift", to_np(dshift), DS)
    check_f32("dscale", to_np(dscale), DC)


def test_forward_is_deterministic_and_bwd_repeatable(pvl):
    x, shift, scale, dy = inputs(1, 500, 5120, seed=11)
    a = run(pvl, x, shift, scale, dy, 1e-6)
    b = run(pvl, x, shift, scale, dy, 1e-6)
    for u, v in zip(a, b):  # no atomics anywhere: bitwise equal
        assert torch.equal(u, v)


def test_full_size(pvl):
    """The measured size (B = 1, N = 64,000, D = 5120): y and dx on sampled
    rows from the oracle row by row, dshift / dscale from the oracle summed
    over row chunks."""
    B, N, D = 1, 64000, 5120
    x, shift, scale, dy = inputs(B, N, D, seed=64)
    y, _, _, dx, dshift, dscale = run(pvl, x, shift, scale, dy, 1e-6)
    rows = np.random.default_rng(3).choice(N, size=64, replace=False)
    Y, _, _ = oracle.adaln_fwd(x[:, rows], shift, scale)
    DX, _, _ = oracle.adaln_bwd(x[:, rows], shift, scale, dy[:, rows])
    check_bf16("y", to_np(y[:, rows]), Y)
    check_bf16("dx", to_np(dx[:, rows]), DX)
    DS = np.zeros((B, D))
    DC = np.zeros((B, D))
    for n0 in range(0, N, 8000):
        _, ds, dc = oracle.adaln_bwd(x[:, n0:n0 + 8000], shift, scale, dy[:, n0:n0 + 8000])
        DS += ds
        DC += dc
    check_f32("dshift", to_np(dshift), DS)
    check_f32("dscale", to_np(dscale), DC)


def test_autograd_wrapper(pvl):
    x, shift, scale, dy = inputs(2, 33, 640, seed=7)
    xc = x.cuda().requires_grad_()
    sc = shift.cuda().requires_grad_()
    cc = scale.cuda().requires_grad_()
    y = pvl.adaln_modulate(xc, sc, cc)
    y.backward(dy.cuda())
    pvl.device_error()
    DX, DS, DC = oracle.adaln_bwd(x, shift, scale, dy)
    check_bf16("dx", to_np(xc.grad), DX)
    check_f32("dshift", to_np(sc.grad), DS)
    check_f32("dscale", to_np(cc.grad), DC)
