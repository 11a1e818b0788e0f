"""Independent checks that pin the fp64 oracle to something other than itself.

Each check takes the oracle module (or a mutant of it, see
test_oracle_mutants.py) and raises AssertionError when the oracle disagrees
with:
- a brute-force per-pair evaluation of the masked softmax written with plain
  Python loops (no numpy, no grouping by id);
- central finite differences of f = <dO, O(q, k, v)>;
- torch fp64 autograd of the dense masked formula;
- torch's scaled_dot_product_attention on one unpadded episode;
- closed forms (zero keys, constant values) and the packed == separate
  invariant of "lingbot_va_packing" §3.1 (packed batch vs single forwards).
"""

from __future__ import annotations

import math

import numpy as np
import torch


def rand_case(seed, B=2, L=11, H=2, D=3, n_ids=3, p_pad=0.25):
    """Small fp64 inputs with interleaved ids and padding positions."""
    rng = np.random.default_rng(seed)
    q, k, v, do = (rng.standard_normal((B, L, H, D)) for _ in range(4))
    sid = rng.integers(0, n_ids, size=(B, L)).astype(np.int32)
    sid[rng.random((B, L)) < p_pad] = -1
    sid[:, 0] = 0  # at least one valid id per row
    return q, k, v, do, sid


# ---------------------------------------------------------------- brute force
def brute_fwd(q, k, v, sid, scale):
    """Per-pair loops over one (b, h): q/k/v as nested lists [L][D]."""
    L, D = len(q), len(q[0])
    O = [[0.0] * D for _ in range(L)]
    LSE = [-math.inf] * L
    for i in range(L):
        adm = [j for j in range(L) if sid[i] >= 0 and sid[j] == sid[i]]
        if not adm:
            continue
        s = {j: scale * sum(q[i][d] * k[j][d] for d in range(D)) for j in adm}
        mx = max(s.values())
        LSE[i] = mx + math.log(sum(math.exp(s[j] - mx) for j in adm))
        for d in range(D):
            O[i][d] = sum(math.exp(s[j] - LSE[i]) * v[j][d] for j in adm)
    return O, LSE


def check_brute_force(oracle, seed=0, **kw):
    q, k, v, do, sid = rand_case(seed, **kw)
    B, L, H, D = q.shape
    scale = 0.7  # deliberately not 1/sqrt(D)
    O, LSE = oracle.attention_fwd(q, k, v, sid, scale=scale)
    for b in range(B):
        for h in range(H):
            Ob, Lb = brute_fwd(q[b, :, h].tolist(), k[b, :, h].tolist(), v[b, :, h].tolist(),
                               sid[b].tolist(), scale)
            np.testing.assert_allclose(O[b, :, h], np.array(Ob), rtol=0, atol=1e-12)
            np.testing.assert_array_equal(np.isinf(LSE[b, h]), np.isinf(np.array(Lb)))
            fin = np.isfinite(np.array(Lb))
            np.testing.assert_allclose(LSE[b, h][fin], np.array(Lb)[fin], rtol=0, atol=1e-12)


# --------------------------------------------------------- finite differences
def check_finite_differences(oracle, seed=1, eps=1e-6, **kw):
    kw = {"B": 1, "L": 9, "H": 2, "D": 3, **kw}
    q, k, v, do, sid = rand_case(seed, **kw)
    scale = 0.9
    dQ, dK, dV, _ = oracle.attention_bwd(q, k, v, do, sid, scale=scale)

    def f(qq, kk, vv):
        O, _ = oracle.attention_fwd(qq, kk, vv, sid, scale=scale)
        return float((O * do).sum())

    inputs = {"q": q, "k": k, "v": v}
    for name, g in (("q", dQ), ("k", dK), ("v", dV)):
        x = inputs[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            plus = dict(inputs)
            minus = dict(inputs)
            plus[name] = x.copy()
            minus[name] = x.copy()
            plus[name][idx] += eps
            minus[name][idx] -= eps
            num[idx] = (f(plus["q"], plus["k"], plus["v"])
                        - f(minus["q"], minus["k"], minus["v"])) / (2 * eps)
        err = np.abs(num - g).max() / max(1.0, np.abs(num).max())
        assert err < 1e-6, f"d{name}: finite-difference mismatch {err:.3e}"


# ------------------------------------------------------- torch fp64 autograd
def torch_dense(q, k, v, sid, scale):
    """Dense masked attention in torch fp64; rows with no admissible key give 0."""
    S = scale * torch.einsum("bihd,bjhd->bhij", q, k)
    sid = torch.as_tensor(sid)
    M = (sid[:, :, None] == sid[:, None, :]) & (sid[:, :, None] >= 0)  # [B, i, j]
    M = M[:, None]
    S = torch.where(M, S, torch.full_like(S, -1e300))
    P = torch.softmax(S, dim=-1) * M
    O = torch.einsum("bhij,bjhd->bihd", P, v)
    lse = torch.where(M.any(-1), torch.logsumexp(S, dim=-1), torch.full_like(S[..., 0], -math.inf))
    return O, lse


def check_torch_autograd(oracle, seed=2, **kw):
    kw = {"B": 2, "L": 40, "H": 2, "D": 8, "n_ids": 4, **kw}
    q, k, v, do, sid = rand_case(seed, **kw)
    scale = 1.0 / math.sqrt(q.shape[-1])
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    O_t, lse_t = torch_dense(tq, tk, tv, sid, scale)
    (O_t * torch.tensor(do)).sum().backward()
    O, LSE = oracle.attention_fwd(q, k, v, sid)
    dQ, dK, dV, _ = oracle.attention_bwd(q, k, v, do, sid)
    np.testing.assert_allclose(O, O_t.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, lse_t.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dQ, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dK, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dV, tv.grad.numpy(), rtol=0, atol=1e-12)


def check_sdpa_single_episode(oracle, seed=3, L=200, H=3, D=16):
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((1, L, H, D)) for _ in range(3))
    sid = np.zeros((1, L), np.int32)
    O, _ = oracle.attention_fwd(q, k, v, sid)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.tensor(x).permute(0, 2, 1, 3) for x in (q, k, v))).permute(0, 2, 1, 3)
    np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)


# ------------------------------------------------------------- closed forms
def check_closed_forms(oracle, seed=4):
    q, k, v, do, sid = rand_case(seed, B=2, L=30, H=2, D=5, n_ids=3)
    # zero keys: uniform P over the admissible set
    O, LSE = oracle.attention_fwd(q, np.zeros_like(k), v, sid)
    for b in range(sid.shape[0]):
        for i in range(sid.shape[1]):
            if sid[b, i] < 0:
                assert np.all(O[b, i] == 0) and np.all(np.isneginf(LSE[b, :, i]))
                continue
            adm = sid[b] == sid[b, i]
            np.testing.assert_allclose(LSE[b, :, i], math.log(adm.sum()), rtol=0, atol=1e-13)
            np.testing.assert_allclose(O[b, i], v[b, adm].mean(axis=0), rtol=0, atol=1e-13)
    # constant values: O = that value on every valid row
    c = np.broadcast_to(np.arange(5.0)[None, None, None, :] - 2.0, v.shape).copy()
    O, _ = oracle.attention_fwd(q, k, c, sid)
    valid = sid >= 0
    np.testing.assert_allclose(O[valid], c[valid], rtol=0, atol=1e-13)


def check_delta_identity(oracle, seed=5):
    q, k, v, do, sid = rand_case(seed, B=2, L=25, H=2, D=4)
    O, _ = oracle.attention_fwd(q, k, v, sid)
    _, _, _, Delta = oracle.attention_bwd(q, k, v, do, sid)
    np.testing.assert_allclose(Delta, np.einsum("blhd,blhd->bhl", do, O), rtol=0, atol=1e-12)


# ------------------------------------------------- packed == separate, padding
def check_packed_equals_separate(oracle, seed=6):
    """Row 0: three episodes concatenated with padding between and after them;
    row 1: one episode zero-padded at the end (the two packing forms)."""
    rng = np.random.default_rng(seed)
    B, L, H, D = 2, 48, 2, 4
    q, k, v, do = (rng.standard_normal((B, L, H, D)) for _ in range(4))
    sid = np.full((B, L), -1, np.int32)
    spans = [(0, 0, 10, 0), (0, 12, 25, 1), (0, 25, 40, 2), (1, 0, 31, 3)]
    for b, a, e, s in spans:
        sid[b, a:e] = s
    O, LSE = oracle.attention_fwd(q, k, v, sid)
    dQ, dK, dV, _ = oracle.attention_bwd(q, k, v, do, sid)
    for b, a, e, _ in spans:
        sl = slice(a, e)
        one = np.zeros((1, e - a), np.int32)
        Os, Ls = oracle.attention_fwd(q[b:b + 1, sl], k[b:b + 1, sl], v[b:b + 1, sl], one)
        gs = oracle.attention_bwd(q[b:b + 1, sl], k[b:b + 1, sl], v[b:b + 1, sl],
                                  do[b:b + 1, sl], one)
        np.testing.assert_allclose(O[b, sl], Os[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE[b, :, sl], Ls[0], rtol=0, atol=1e-12)
        for full, sep in zip((dQ, dK, dV), gs[:3]):
            np.testing.assert_allclose(full[b, sl], sep[0], rtol=0, atol=1e-12)
    pad = sid < 0
    assert np.all(O[pad] == 0.0) and np.all(dQ[pad] == 0.0)
    assert np.all(dK[pad] == 0.0) and np.all(dV[pad] == 0.0)
    assert np.all(np.isneginf(LSE.transpose(0, 2, 1)[pad]))
    assert np.isfinite(O).all() and np.isfinite(dQ).all()


ALL_PINS = [
    check_brute_force,
    check_finite_differences,
    check_torch_autograd,
    check_sdpa_single_episode,
    check_closed_forms,
    check_delta_identity,
    check_packed_equals_separate,
]
