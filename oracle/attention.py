"""Oracle: seq_id-masked softmax attention and its gradient, fp64 on the CPU.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition ("furniture_packing_variable_length", attention masking: tokens
attend only to tokens with the same seq_id, and seq_id -1 is out on both the
query and the key side; "lingbot_va_attn_profiling", packing proposal: the
mask condition doc_id[q] == doc_id[k]).  Per batch row b and head h, with the
inputs exactly as handed to the kernels (bf16 values upcast to fp64):

    M_ij   = [s_i == s_j and s_i >= 0]
    S_ij   = scale * <q_i, k_j>
    LSE_i  = log sum_{j : M_ij} exp(S_ij)          (natural log)
    P_ij   = M_ij * exp(S_ij - LSE_i)
    O_i    = sum_j P_ij v_j

    dP_ij  = <dO_i, v_j>
    Delta_i = sum_j P_ij dP_ij
    dS_ij  = P_ij (dP_ij - Delta_i)
    dQ_i   = scale * sum_j dS_ij k_j
    dK_j   = scale * sum_i dS_ij q_i
    dV_j   = sum_i P_ij dO_i

A query with s_i = -1 has no admissible key: O_i = 0, LSE_i = -inf, dQ_i = 0.
A key with s_j = -1 is never admissible: dK_j = dV_j = 0.  The pages fix no
softmax scale; the default is 1 / sqrt(D).

Cross attention ("lingbot_va_packing" §2.1: the latent and the action tokens
carry their own seq_ids, and frames past an episode's valid length drop out
of the self and of the cross attention mask): queries q [B, Lq] with ids s_i
and keys k, v [B, Lk] with their own ids t_j, M_ij = [s_i == t_j and
s_i >= 0]; everything else is as above.  A valid query whose id has no key
gets O_i = 0, LSE_i = -inf, dQ_i = 0, like a padding row.  Self attention is
the case t = s (k_seq_id omitted).

The sums over {j : M_ij} are evaluated by enumerating that set: for each id
s >= 0 the positions holding s form the query rows and the key columns of one
dense softmax.  Query rows are taken ``block`` at a time (summation order only).
The LSE uses the usual max subtraction.  numpy matmul is the only library step.
"""

from __future__ import annotations

import math

import numpy as np


def _f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _groups(seq_row: np.ndarray):
    """(id, positions) for every id >= 0 present in one row."""
    seq_row = np.asarray(seq_row)
    for s in np.unique(seq_row[seq_row >= 0]):
        yield int(s), np.nonzero(seq_row == s)[0]


def _check(q, k, seq_id, k_seq_id):
    if len(q.shape) != 4 or len(k.shape) != 4:
        raise ValueError("expected [B, L, H, D]")
    B, Lq, H, D = q.shape
    if k.shape[0] != B or k.shape[2] != H or k.shape[3] != D:
        raise ValueError("q and k differ in B, H or D")
    if tuple(np.asarray(seq_id).shape) != (B, Lq):
        raise ValueError("seq_id must be [B, Lq]")
    if tuple(np.asarray(k_seq_id).shape) != (B, k.shape[1]):
        raise ValueError("k_seq_id must be [B, Lk]")


def _pairs(q_row: np.ndarray, k_row: np.ndarray):
    """(query positions, key positions) for every id >= 0 of the query row."""
    for s, rows in _groups(q_row):
        yield rows, np.nonzero(np.asarray(k_row) == s)[0]


def attention_fwd(q, k, v, seq_id, scale: float | None = None, heads=None, block: int = 512, k_seq_id=None):
    """Returns (O [B, Lq, nh, D], LSE [B, nh, Lq]) in fp64 for the listed heads."""
    k_seq_id = seq_id if k_seq_id is None else k_seq_id
    _check(q, k, seq_id, k_seq_id)
    B, L, H, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    heads = list(range(H)) if heads is None else list(heads)
    seq_id, k_seq_id = np.asarray(seq_id), np.asarray(k_seq_id)
    O = np.zeros((B, L, len(heads), D))
    LSE = np.full((B, len(heads), L), -np.inf)
    for b in range(B):
        for hi, h in enumerate(heads):
            qb, kb, vb = _f64(q[b, :, h]), _f64(k[b, :, h]), _f64(v[b, :, h])
            for idx, kidx in _pairs(seq_id[b], k_seq_id[b]):
                if len(kidx) == 0:
                    continue  # no admissible key: O = 0, LSE = -inf
                Ks, Vs = kb[kidx], vb[kidx]
                for i0 in range(0, len(idx), block):
                    rows = idx[i0:i0 + block]
                    S = scale * (qb[rows] @ Ks.T)
                    m = S.max(axis=1)
                    lse = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
                    P = np.exp(S - lse[:, None])
                    O[b, rows, hi] = P @ Vs
                    LSE[b, hi, rows] = lse
    return O, LSE


def attention_bwd(q, k, v, do, seq_id, scale: float | None = None, heads=None, block: int = 512, k_seq_id=None):
    """Returns (dQ [B, Lq, nh, D], dK, dV [B, Lk, nh, D], Delta [B, nh, Lq]) in
    fp64 for the listed heads.

    Recomputes P from its own LSE; nothing produced by a kernel enters here.
    """
    k_seq_id = seq_id if k_seq_id is None else k_seq_id
    _check(q, k, seq_id, k_seq_id)
    B, L, H, D = q.shape
    Lk = k.shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    heads = list(range(H)) if heads is None else list(heads)
    seq_id, k_seq_id = np.asarray(seq_id), np.asarray(k_seq_id)
    dQ = np.zeros((B, L, len(heads), D))
    dK = np.zeros((B, Lk, len(heads), D))
    dV = np.zeros((B, Lk, len(heads), D))
    Delta = np.zeros((B, len(heads), L))
    for b in range(B):
        for hi, h in enumerate(heads):
            qb, kb, vb, dob = _f64(q[b, :, h]), _f64(k[b, :, h]), _f64(v[b, :, h]), _f64(do[b, :, h])
            for idx, kidx in _pairs(seq_id[b], k_seq_id[b]):
                if len(kidx) == 0:
                    continue  # no admissible key: dQ = 0, Delta = 0
                Ks, Vs = kb[kidx], vb[kidx]
                dKs = np.zeros_like(Ks)
                dVs = np.zeros_like(Vs)
                for i0 in range(0, len(idx), block):
                    rows = idx[i0:i0 + block]
                    S = scale * (qb[rows] @ Ks.T)
                    m = S.max(axis=1)
                    lse = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
                    P = np.exp(S - lse[:, None])
                    dP = dob[rows] @ Vs.T
                    delta = (P * dP).sum(axis=1)
                    dS = P * (dP - delta[:, None])
                    dQ[b, rows, hi] = scale * (dS @ Ks)
                    dKs += scale * (dS.T @ qb[rows])
                    dVs += P.T @ dob[rows]
                    Delta[b, hi, rows] = delta
                dK[b, kidx, hi] = dKs
                dV[b, kidx, hi] = dVs
    return dQ, dK, dV, Delta


def effective_pairs(seq_id, k_seq_id=None) -> int:
    """Admissible (query, key) pairs per head: sum over rows and ids of
    (queries with the id) * (keys with the id); n_id^2 for self attention."""
    seq_id = np.asarray(seq_id)
    k_seq_id = seq_id if k_seq_id is None else np.asarray(k_seq_id)
    total = 0
    for b in range(seq_id.shape[0]):
        for idx, kidx in _pairs(seq_id[b], k_seq_id[b]):
            total += len(idx) * len(kidx)
    return total
