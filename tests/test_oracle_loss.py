"""The fp64 frame_valid loss oracle against independent checks (CPU only):
a per-element brute force of the pages' definition, torch's own mse_loss on
the masked elements and its autograd, central finite differences, closed
forms, the packed == separate invariant, the seq_id route to the same mask,
and planted mistakes that the checks must catch."""

import os
import types

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "loss.py")


def case(seed, B=3, F=5, T=4, C=6):
    rng = np.random.default_rng(seed)
    valid_frames = rng.integers(0, F + 1, size=B)
    valid_frames[0] = F          # one row fully valid
    valid_frames[1] = min(valid_frames[1], F - 1)  # one row with padding frames
    pred = rng.standard_normal((B, F * T, C))
    target = rng.standard_normal((B, F * T, C))
    return pred, target, valid_frames, F, T


def check_brute_force(mod, seed=0):
    """Every element visited in Python loops, the frame of token n being n // T."""
    pred, target, vf, F, T = case(seed)
    B, L, C = pred.shape
    s, n = 0.0, 0
    for b in range(B):
        for tok in range(L):
            if tok // T < vf[b]:
                n += 1
                for c in range(C):
                    s += (pred[b, tok, c] - target[b, tok, c]) ** 2
    valid = mod.frame_valid_tokens(vf, F, T)
    loss, n_valid = mod.masked_mse(pred, target, valid)
    assert n_valid == n
    assert abs(loss - s / (C * n)) <= 1e-12 * max(1.0, s / (C * n))
    g = mod.masked_mse_grad(pred, target, valid)
    for b in range(B):
        for tok in range(L):
            exp = 2 * (pred[b, tok] - target[b, tok]) / (C * n) if tok // T < vf[b] else np.zeros(C)
            np.testing.assert_allclose(g[b, tok], exp, rtol=0, atol=1e-15)


def check_torch(mod, seed=1):
    """The page's own formulation in torch: frame_valid = arange(F) < valid_frames[:, None],
    expanded over the frame's tokens, mse_loss over the selected elements."""
    pred, target, vf, F, T = case(seed)
    B, L, C = pred.shape
    tp = torch.tensor(pred, requires_grad=True)
    tt = torch.tensor(target)
    frame_valid = torch.arange(F)[None, :] < torch.tensor(vf)[:, None]
    tok_valid = frame_valid[:, :, None].expand(B, F, T).reshape(B, L)
    ref = torch.nn.functional.mse_loss(tp[tok_valid], tt[tok_valid])
    ref.backward(torch.tensor(0.75, dtype=torch.float64))
    valid = mod.frame_valid_tokens(vf, F, T)
    loss, _ = mod.masked_mse(pred, target, valid)
    assert abs(loss - ref.item()) <= 1e-13
    np.testing.assert_allclose(mod.masked_mse_grad(pred, target, valid, dloss=0.75), tp.grad.numpy(),
                               rtol=0, atol=1e-15)


def check_finite_differences(mod, seed=2, h=1e-6):
    pred, target, vf, F, T = case(seed, B=2, F=3, T=2, C=3)
    valid = mod.frame_valid_tokens(vf, F, T)
    g = mod.masked_mse_grad(pred, target, valid)
    num = np.zeros_like(pred)
    for idx in np.ndindex(*pred.shape):
        a, b = pred.copy(), pred.copy()
        a[idx] += h
        b[idx] -= h
        num[idx] = (mod.masked_mse(a, target, valid)[0] - mod.masked_mse(b, target, valid)[0]) / (2 * h)
    assert np.abs(num - g).max() < 1e-8


def check_closed_forms(mod):
    rng = np.random.default_rng(3)
    B, F, T, C = 2, 4, 3, 5
    L = F * T
    p = rng.standard_normal((B, L, C))
    # prediction equal to the target: zero loss, zero gradient
    valid = mod.frame_valid_tokens([2, 4], F, T)
    loss, n = mod.masked_mse(p, p.copy(), valid)
    assert loss == 0.0 and n == (2 + 4) * T
    assert not mod.masked_mse_grad(p, p.copy(), valid).any()
    # every frame valid: the plain mean squared error
    t = rng.standard_normal((B, L, C))
    full = mod.frame_valid_tokens([F, F], F, T)
    assert abs(mod.masked_mse(p, t, full)[0] - float(((p - t) ** 2).mean())) < 1e-13
    # a constant difference d on the valid tokens: loss d^2, whatever the padding holds
    t2 = p - 0.5
    t2[~valid] = 1e6
    assert abs(mod.masked_mse(p, t2, valid)[0] - 0.25) < 1e-14
    g = mod.masked_mse_grad(p, t2, valid)
    assert not g[~valid].any()
    np.testing.assert_allclose(g[valid], 2 * 0.5 / (C * valid.sum()), rtol=1e-14)
    # no valid frame: loss 0, gradient 0
    none = mod.frame_valid_tokens([0, 0], F, T)
    assert mod.masked_mse(p, t, none) == (0.0, 0)
    assert not mod.masked_mse_grad(p, t, none).any()
    # the mask itself: frame f of row b valid iff f < valid_frames[b]
    m = mod.frame_valid_tokens([1, 3], F, T)
    assert m[0].tolist() == [True] * T + [False] * (3 * T)
    assert m[1].tolist() == [True] * (3 * T) + [False] * T


def check_packed_equals_separate(mod, seed=4):
    """The padded batch's loss is the valid-token-weighted mean of the
    episodes' own unpadded losses ("lingbot_va_packing" §3.1: packed and
    separate losses agree)."""
    pred, target, vf, F, T = case(seed, B=4, F=6, T=3, C=4)
    valid = mod.frame_valid_tokens(vf, F, T)
    loss, n = mod.masked_mse(pred, target, valid)
    num, den = 0.0, 0
    for b in range(pred.shape[0]):
        k = int(vf[b]) * T
        if k == 0:
            continue
        e, ne = mod.masked_mse(pred[b:b + 1, :k], target[b:b + 1, :k], np.ones((1, k), dtype=bool))
        assert ne == k
        num += e * k
        den += k
    assert den == n
    assert abs(loss - num / den) < 1e-13


def check_seq_id_route(mod):
    """On pad-collated rows (one episode per row) the attention's seq_ids give
    the same token mask as frame_valid."""
    vf = np.array([3, 5, 0, 2])
    F, T = 5, 4
    seq = oracle.build_seq_ids(np.full((4, 1), F), vf[:, None], T, F * T)
    np.testing.assert_array_equal(mod.valid_from_seq_id(seq), mod.frame_valid_tokens(vf, F, T))


CHECKS = [check_brute_force, check_torch, check_finite_differences, check_closed_forms,
          check_packed_equals_separate, check_seq_id_route]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_check(check):
    check(oracle.loss)


MUTATIONS = {
    "mean_over_all_tokens": ("n_valid = int(valid.sum())\n    if n_valid == 0:\n        return 0.0, 0",
                             "n_valid = int(valid.size)\n    if n_valid == 0:\n        return 0.0, 0"),
    "no_channel_divisor": ("return float((diff * diff).sum() / (C * n_valid)), n_valid",
                           "return float((diff * diff).sum() / n_valid), n_valid"),
    "frame_valid_le": ("frame_valid = np.arange(F)[None, :] < valid_frames[:, None]",
                       "frame_valid = np.arange(F)[None, :] <= valid_frames[:, None]"),
    "mask_tiled_not_repeated": ("return np.repeat(frame_valid, T, axis=1)", "return np.tile(frame_valid, (1, T))"),
    "grad_without_two": ("g[valid] = (2.0 * float(dloss) / (C * n_valid)) * (p - t)[valid]",
                         "g[valid] = (float(dloss) / (C * n_valid)) * (p - t)[valid]"),
    "grad_on_padding": ("g[valid] = (2.0 * float(dloss) / (C * n_valid)) * (p - t)[valid]",
                        "g[:] = (2.0 * float(dloss) / (C * n_valid)) * (p - t)"),
    "grad_sign": ("g[valid] = (2.0 * float(dloss) / (C * n_valid)) * (p - t)[valid]",
                  "g[valid] = (2.0 * float(dloss) / (C * n_valid)) * (t - p)[valid]"),
    "seq_id_mask_gt": ("return np.asarray(seq_id) >= 0", "return np.asarray(seq_id) > 0"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_checks_catch_mutant(name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType("loss_mutant")
    exec(compile(src.replace(old, new), "loss_mutant", "exec"), mod.__dict__)
    caught = []
    for check in CHECKS:
        try:
            check(mod)
        except (AssertionError, ValueError, IndexError):
            caught.append(check.__name__)
    assert caught, f"no check caught {name}"
