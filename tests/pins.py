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
The same checks run on cross attention (query and key ids and lengths
differ, "lingbot_va_packing" §2.1), including ids that only one side holds.
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


def rand_cross_case(seed, B=2, Lq=11, Lk=7, H=2, D=3, n_ids=4, p_pad=0.25):
    """Small fp64 cross-attention inputs: query and key ids drawn separately,
    so some ids have queries but no keys and the other way round."""
    rng = np.random.default_rng(seed)
    q, do = (rng.standard_normal((B, Lq, H, D)) for _ in range(2))
    k, v = (rng.standard_normal((B, Lk, H, D)) for _ in range(2))
    qsid = rng.integers(0, n_ids, size=(B, Lq)).astype(np.int32)
    ksid = rng.integers(0, n_ids - 1, size=(B, Lk)).astype(np.int32)  # id n_ids-1: queries only
    qsid[rng.random((B, Lq)) < p_pad] = -1
    ksid[rng.random((B, Lk)) < p_pad] = -1
    qsid[:, 0] = 0
    ksid[:, 0] = 0  # at least one admissible pair per row
    return q, k, v, do, qsid, ksid


# ---------------------------------------------------------------- brute force
def brute_fwd(q, k, v, sid, scale, ksid=None):
    """Per-pair loops over one (b, h): q as nested lists [Lq][D], k/v [Lk][D]."""
    ksid = sid if ksid is None else ksid
    L, D = len(q), len(q[0])
    O = [[0.0] * D for _ in range(L)]
    LSE = [-math.inf] * L
    for i in range(L):
        adm = [j for j in range(len(k)) if sid[i] >= 0 and ksid[j] == sid[i]]
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


def check_brute_force_cross(oracle, seed=20):
    q, k, v, do, qsid, ksid = rand_cross_case(seed)
    B, L, H, D = q.shape
    scale = 0.6
    O, LSE = oracle.attention_fwd(q, k, v, qsid, scale=scale, k_seq_id=ksid)
    assert O.shape == q.shape and LSE.shape == (B, H, L)
    for b in range(B):
        for h in range(H):
            Ob, Lb = brute_fwd(q[b, :, h].tolist(), k[b, :, h].tolist(), v[b, :, h].tolist(),
                               qsid[b].tolist(), scale, ksid[b].tolist())
            np.testing.assert_allclose(O[b, :, h], np.array(Ob), rtol=0, atol=1e-12)
            np.testing.assert_array_equal(np.isinf(LSE[b, h]), np.isinf(np.array(Lb)))
            fin = np.isfinite(np.array(Lb))
            np.testing.assert_allclose(LSE[b, h][fin], np.array(Lb)[fin], rtol=0, atol=1e-12)


# --------------------------------------------------------- finite differences
def check_finite_differences_cross(oracle, seed=21, eps=1e-6):
    q, k, v, do, qsid, ksid = rand_cross_case(seed, B=1, Lq=6, Lk=5, H=1, D=3)
    scale = 0.8
    dQ, dK, dV, _ = oracle.attention_bwd(q, k, v, do, qsid, scale=scale, k_seq_id=ksid)
    assert dQ.shape == q.shape and dK.shape == k.shape and dV.shape == v.shape

    def f(qq, kk, vv):
        O, _ = oracle.attention_fwd(qq, kk, vv, qsid, scale=scale, k_seq_id=ksid)
        return float((O * do).sum())

    inputs = {"q": q, "k": k, "v": v}
    for name, g in (("q", dQ), ("k", dK), ("v", dV)):
        x = inputs[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            plus, minus = dict(inputs), dict(inputs)
            plus[name], minus[name] = x.copy(), x.copy()
            plus[name][idx] += eps
            minus[name][idx] -= eps
            num[idx] = (f(plus["q"], plus["k"], plus["v"]) - f(minus["q"], minus["k"], minus["v"])) / (2 * eps)
        err = np.abs(num - g).max() / max(1.0, np.abs(num).max())
        assert err < 1e-6, f"cross d{name}: finite-difference mismatch {err:.3e}"


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
def torch_dense(q, k, v, sid, scale, ksid=None):
    """Dense masked attention in torch fp64; rows with no admissible key give 0."""
    S = scale * torch.einsum("bihd,bjhd->bhij", q, k)
    sid = torch.as_tensor(sid)
    ksid = sid if ksid is None else torch.as_tensor(ksid)
    M = (sid[:, :, None] == ksid[:, None, :]) & (sid[:, :, None] >= 0)  # [B, i, j]
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


def check_torch_autograd_cross(oracle, seed=22):
    q, k, v, do, qsid, ksid = rand_cross_case(seed, B=2, Lq=37, Lk=23, H=2, D=8, n_ids=5)
    scale = 1.0 / math.sqrt(q.shape[-1])
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    O_t, lse_t = torch_dense(tq, tk, tv, qsid, scale, ksid)
    (O_t * torch.tensor(do)).sum().backward()
    O, LSE = oracle.attention_fwd(q, k, v, qsid, k_seq_id=ksid)
    dQ, dK, dV, _ = oracle.attention_bwd(q, k, v, do, qsid, k_seq_id=ksid)
    np.testing.assert_allclose(O, O_t.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, lse_t.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dQ, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dK, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dV, tv.grad.numpy(), rtol=0, atol=1e-12)


def check_sdpa_cross_single_episode(oracle, seed=23, Lq=150, Lk=70, H=2, D=16):
    """One episode on each side, no padding: plain (unmasked) cross attention."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, Lq, H, D))
    k, v = (rng.standard_normal((1, Lk, H, D)) for _ in range(2))
    O, _ = oracle.attention_fwd(q, k, v, np.zeros((1, Lq), np.int32), k_seq_id=np.zeros((1, Lk), np.int32))
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.tensor(x).permute(0, 2, 1, 3) for x in (q, k, v))).permute(0, 2, 1, 3)
    np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)


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


def check_closed_forms_cross(oracle, seed=24):
    """Zero keys: uniform P over the keys with the query's id, LSE = log of
    their number; a valid query whose id has no key behaves like padding."""
    q, k, v, do, qsid, ksid = rand_cross_case(seed, B=2, Lq=29, Lk=17, H=2, D=4, n_ids=4)
    O, LSE = oracle.attention_fwd(q, np.zeros_like(k), v, qsid, k_seq_id=ksid)
    dQ, _, _, _ = oracle.attention_bwd(q, k, v, do, qsid, k_seq_id=ksid)
    seen_keyless = False
    for b in range(qsid.shape[0]):
        for i in range(qsid.shape[1]):
            adm = (ksid[b] == qsid[b, i]) & (qsid[b, i] >= 0)
            if not adm.any():
                seen_keyless |= qsid[b, i] >= 0
                assert np.all(O[b, i] == 0) and np.all(np.isneginf(LSE[b, :, i])) and np.all(dQ[b, i] == 0)
                continue
            np.testing.assert_allclose(LSE[b, :, i], math.log(adm.sum()), rtol=0, atol=1e-13)
            np.testing.assert_allclose(O[b, i], v[b, adm].mean(axis=0), rtol=0, atol=1e-13)
    assert seen_keyless  # the case carries valid queries without keys


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


def check_packed_equals_separate_cross(oracle, seed=25):
    """Episodes packed on both sides with different lengths per side (query
    spans and key spans of each id), padding between and after them."""
    rng = np.random.default_rng(seed)
    B, Lq, Lk, H, D = 2, 40, 26, 2, 4
    q, do = (rng.standard_normal((B, Lq, H, D)) for _ in range(2))
    k, v = (rng.standard_normal((B, Lk, H, D)) for _ in range(2))
    qsid = np.full((B, Lq), -1, np.int32)
    ksid = np.full((B, Lk), -1, np.int32)
    spans = [(0, (0, 9), (0, 5), 0), (0, (11, 24), (6, 14), 1), (0, (24, 37), (14, 20), 2),
             (1, (0, 30), (2, 25), 3)]
    for b, (qa, qe), (ka, ke), s in spans:
        qsid[b, qa:qe] = s
        ksid[b, ka:ke] = s
    O, LSE = oracle.attention_fwd(q, k, v, qsid, k_seq_id=ksid)
    dQ, dK, dV, _ = oracle.attention_bwd(q, k, v, do, qsid, k_seq_id=ksid)
    for b, (qa, qe), (ka, ke), _ in spans:
        qs, ks = slice(qa, qe), slice(ka, ke)
        z_q, z_k = np.zeros((1, qe - qa), np.int32), np.zeros((1, ke - ka), np.int32)
        Os, Ls = oracle.attention_fwd(q[b:b + 1, qs], k[b:b + 1, ks], v[b:b + 1, ks], z_q, k_seq_id=z_k)
        gs = oracle.attention_bwd(q[b:b + 1, qs], k[b:b + 1, ks], v[b:b + 1, ks], do[b:b + 1, qs], z_q,
                                  k_seq_id=z_k)
        np.testing.assert_allclose(O[b, qs], Os[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE[b, :, qs], Ls[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dQ[b, qs], gs[0][0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dK[b, ks], gs[1][0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dV[b, ks], gs[2][0], rtol=0, atol=1e-12)
    assert np.all(O[qsid < 0] == 0.0) and np.all(dQ[qsid < 0] == 0.0)
    assert np.all(dK[ksid < 0] == 0.0) and np.all(dV[ksid < 0] == 0.0)


ALL_PINS = [
    check_brute_force,
    check_finite_differences,
    check_torch_autograd,
    check_sdpa_single_episode,
    check_closed_forms,
    check_delta_identity,
    check_packed_equals_separate,
    check_brute_force_cross,
    check_finite_differences_cross,
    check_torch_autograd_cross,
    check_sdpa_cross_single_episode,
    check_closed_forms_cross,
    check_packed_equals_separate_cross,
]
