"""The fp64 LayerNorm-Modulate oracle against independent checks (CPU only):
torch fp64 autograd of torch's own layer_norm, central finite differences,
closed forms, and planted mistakes that the checks must catch."""

import math
import os
import types

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "adaln.py")


def case(seed, B=2, N=7, D=12, scale_amp=0.5):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, N, D)) * 3.0 + rng.standard_normal((B, N, 1))  # row offsets
    shift = rng.standard_normal((B, D))
    scale = rng.standard_normal((B, D)) * scale_amp
    dy = rng.standard_normal((B, N, D))
    return x, shift, scale, dy


def check_torch(mod, seed=0, eps=1e-6):
    x, shift, scale, dy = case(seed)
    tx, ts, tc = (torch.tensor(a, requires_grad=True) for a in (x, shift, scale))
    y_t = torch.nn.functional.layer_norm(tx, (x.shape[2],), eps=eps) * (1 + tc[:, None, :]) + ts[:, None, :]
    y_t.backward(torch.tensor(dy))
    y, mu, r = mod.adaln_fwd(x, shift, scale, eps=eps)
    dx, dshift, dscale = mod.adaln_bwd(x, shift, scale, dy, eps=eps)
    np.testing.assert_allclose(y, y_t.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(mu, x.mean(axis=2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r, 1 / np.sqrt(x.var(axis=2) + eps), rtol=1e-12, atol=0)
    np.testing.assert_allclose(dx, tx.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dshift, ts.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dscale, tc.grad.numpy(), rtol=0, atol=1e-11)


def check_finite_differences(mod, seed=1, h=1e-6):
    x, shift, scale, dy = case(seed, B=1, N=3, D=5)
    dx, dshift, dscale = mod.adaln_bwd(x, shift, scale, dy)

    def f(xx, ss, cc):
        y, _, _ = mod.adaln_fwd(xx, ss, cc)
        return float((y * dy).sum())

    for name, arr, g in (("x", x, dx), ("shift", shift, dshift), ("scale", scale, dscale)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(*arr.shape):
            a, b = arr.copy(), arr.copy()
            a[idx] += h
            b[idx] -= h
            args_p = {"x": x, "shift": shift, "scale": scale}
            args_m = dict(args_p)
            args_p[name], args_m[name] = a, b
            num[idx] = (f(args_p["x"], args_p["shift"], args_p["scale"])
                        - f(args_m["x"], args_m["shift"], args_m["scale"])) / (2 * h)
        err = np.abs(num - g).max() / max(1.0, np.abs(num).max())
        assert err < 1e-6, f"d{name}: finite-difference mismatch {err:.2e}"


def check_closed_forms(mod):
    rng = np.random.default_rng(2)
    B, N, D = 2, 4, 16
    shift = rng.standard_normal((B, D))
    scale = rng.standard_normal((B, D))
    # constant rows: xh = 0, so y = shift and no gradient flows to x or scale
    x = np.broadcast_to(rng.standard_normal((B, N, 1)), (B, N, D)).copy()
    y, _, _ = mod.adaln_fwd(x, shift, scale)
    np.testing.assert_allclose(y, np.broadcast_to(shift[:, None, :], y.shape), rtol=0, atol=1e-12)
    dy = rng.standard_normal((B, N, D))
    dx, dshift, dscale = mod.adaln_bwd(x, shift, scale, dy)
    np.testing.assert_allclose(dscale, 0.0, atol=1e-12)
    np.testing.assert_allclose(dshift, dy.sum(axis=1), rtol=0, atol=1e-12)
    # zero modulation: each output row has mean 0 and variance var / (var + eps)
    x = rng.standard_normal((B, N, D)) * 5 + 2
    y, _, _ = mod.adaln_fwd(x, np.zeros((B, D)), np.zeros((B, D)), eps=1e-6)
    np.testing.assert_allclose(y.mean(axis=2), 0.0, atol=1e-12)
    v = x.var(axis=2)
    np.testing.assert_allclose(y.var(axis=2), v / (v + 1e-6), rtol=1e-12)
    # a two-value row [a, b]: xh = [-1, 1] (up to eps), so y = shift -/+ (1 + scale)
    x2 = np.array([[[3.0, 7.0]]])
    y2, mu2, r2 = mod.adaln_fwd(x2, np.array([[0.5, -0.5]]), np.array([[1.0, 2.0]]), eps=0.0)
    np.testing.assert_allclose(mu2, [[5.0]], rtol=0, atol=0)
    np.testing.assert_allclose(r2, [[0.5]], rtol=0, atol=0)
    np.testing.assert_allclose(y2, [[[0.5 - 2.0, -0.5 + 3.0]]], rtol=0, atol=1e-15)
    # dy = 0 gives zero gradients
    dx0, ds0, dc0 = mod.adaln_bwd(x, shift, scale, np.zeros_like(x))
    assert not dx0.any() and not ds0.any() and not dc0.any()


CHECKS = [check_torch, check_finite_differences, check_closed_forms]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_check(check):
    check(oracle.adaln)


MUTATIONS = {
    "unbiased_variance": ("var = (xc * xc).mean(axis=2)", "var = (xc * xc).sum(axis=2) / (x.shape[2] - 1)"),
    "eps_outside_sqrt": ("r = 1.0 / np.sqrt(var + eps)", "r = 1.0 / (np.sqrt(var) + eps)"),
    "modulation_without_one": ("y = xh * (1.0 + scale[:, None, :]) + shift[:, None, :]", "y = xh * scale[:, None, :] + shift[:, None, :]"),
    "dx_missing_xh_term": ("dx = r[:, :, None] * (g - mg[:, :, None] - xh * mgx[:, :, None])", "dx = r[:, :, None] * (g - mg[:, :, None])"),
    "dscale_without_xh": ("dscale = (dy * xh).sum(axis=1)", "dscale = dy.sum(axis=1)"),
    "dshift_over_features": ("dshift = dy.sum(axis=1)", "dshift = dy.sum(axis=2)"),
    "g_without_modulation": ("g = dy * (1.0 + scale[:, None, :])", "g = dy"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_checks_catch_mutant(name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType("adaln_mutant")
    exec(compile(src.replace(old, new), "adaln_mutant", "exec"), mod.__dict__)
    caught = []
    for check in CHECKS:
        try:
            check(mod)
        except (AssertionError, ValueError, IndexError):
            caught.append(check.__name__)
    assert caught, f"no check caught {name}"
