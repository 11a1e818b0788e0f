"""Oracle: tile classification of the seq_id mask.  TEST INFRASTRUCTURE ONLY.

"lingbot_va_packing" §2.1-§2.2: FlexAttention builds a block mask from the
seq_ids and skips blocks in which no query may attend any key; the block mask
must describe the same shape in forward and backward.  The pages give no block
size and no classification rule; the rule below is the plain reading of "skip
a block when no pair in it can match, drop the per-element mask when every
pair matches", made checkable from per-tile summaries only:

- a position p of row b is *valid* iff p < L and seq_id[b, p] >= 0 (query
  tiles over the query ids and length, key tiles over the key ids and length;
  for cross attention, "lingbot_va_packing" §2.1, the two differ);
- per tile t (block_m rows for query tiles, block_n for key tiles):
  nv = number of valid positions, lo / hi = min / max id over them;
- (q-tile, k-tile) is EMPTY if nv_q == 0 or nv_k == 0 or hi_q < lo_k or
  hi_k < lo_q; FULL if lo_q == hi_q == lo_k == hi_k and both tiles are wholly
  valid (nv equals the block size, which also places them wholly inside L);
  PARTIAL otherwise.  Codes: EMPTY 0, PARTIAL 1, FULL 2.

Also produced, as the kernels consume them:
- per query tile the non-empty key tiles, FULL ones first then PARTIAL ones,
  each group in ascending tile index (row_list), with counts row_count and
  row_full; unused list slots hold -1;
- the same per key tile over query tiles (col_list, col_count, col_full);
- q_order / k_order: flat tile indices b * nT + t sorted by descending
  non-empty count, ties by ascending flat index (longest work first).
"""

from __future__ import annotations

import numpy as np

EMPTY, PARTIAL, FULL = 0, 1, 2


def tile_stats(seq_id_row: np.ndarray, L: int, block: int):
    """(nv, lo, hi) per tile of one row; lo = hi = 0 for a tile with nv = 0."""
    n_tiles = -(-L // block)
    nv = np.zeros(n_tiles, np.int32)
    lo = np.zeros(n_tiles, np.int32)
    hi = np.zeros(n_tiles, np.int32)
    for t in range(n_tiles):
        ids = [int(s) for s in seq_id_row[t * block:min((t + 1) * block, L)] if s >= 0]
        nv[t] = len(ids)
        if ids:
            lo[t] = min(ids)
            hi[t] = max(ids)
    return nv, lo, hi


def _classify(nvq, loq, hiq, bm, nvk, lok, hik, bn) -> int:
    if nvq == 0 or nvk == 0 or hiq < lok or hik < loq:
        return EMPTY
    if loq == hiq == lok == hik and nvq == bm and nvk == bn:
        return FULL
    return PARTIAL


def _lists(cls2d: np.ndarray):
    """Compacted non-empty indices along axis 1 of a [n, m] class matrix."""
    n, m = cls2d.shape
    lst = np.full((n, m), -1, np.int32)
    cnt = np.zeros(n, np.int32)
    nfull = np.zeros(n, np.int32)
    for i in range(n):
        full = [j for j in range(m) if cls2d[i, j] == FULL]
        part = [j for j in range(m) if cls2d[i, j] == PARTIAL]
        lst[i, :len(full) + len(part)] = full + part
        cnt[i] = len(full) + len(part)
        nfull[i] = len(full)
    return lst, cnt, nfull


def _longest_first(counts_flat: np.ndarray) -> np.ndarray:
    keys = [(-int(c), i) for i, c in enumerate(counts_flat)]
    return np.array([i for _, i in sorted(keys)], dtype=np.int32)


def build_tile_map(seq_id: np.ndarray, L: int, block_m: int = 128, block_n: int = 128,
                   k_seq_id: np.ndarray | None = None, Lk: int | None = None) -> dict:
    """Tile map of queries (seq_id, length L) against keys (k_seq_id, length
    Lk; the queries' own when omitted)."""
    seq_id = np.asarray(seq_id)
    k_seq_id = seq_id if k_seq_id is None else np.asarray(k_seq_id)
    Lk = L if Lk is None else int(Lk)
    B = seq_id.shape[0]
    nTq = -(-L // block_m)
    nTk = -(-Lk // block_n)
    cls = np.zeros((B, nTq, nTk), np.uint8)
    q_nv = np.zeros((B, nTq), np.int32)
    q_lo = np.zeros((B, nTq), np.int32)
    q_hi = np.zeros((B, nTq), np.int32)
    k_nv = np.zeros((B, nTk), np.int32)
    k_lo = np.zeros((B, nTk), np.int32)
    k_hi = np.zeros((B, nTk), np.int32)
    row_list = np.zeros((B, nTq, nTk), np.int32)
    row_count = np.zeros((B, nTq), np.int32)
    row_full = np.zeros((B, nTq), np.int32)
    col_list = np.zeros((B, nTk, nTq), np.int32)
    col_count = np.zeros((B, nTk), np.int32)
    col_full = np.zeros((B, nTk), np.int32)
    for b in range(B):
        q_nv[b], q_lo[b], q_hi[b] = tile_stats(seq_id[b], L, block_m)
        k_nv[b], k_lo[b], k_hi[b] = tile_stats(k_seq_id[b], Lk, block_n)
        for qt in range(nTq):
            for kt in range(nTk):
                cls[b, qt, kt] = _classify(q_nv[b, qt], q_lo[b, qt], q_hi[b, qt], block_m,
                                           k_nv[b, kt], k_lo[b, kt], k_hi[b, kt], block_n)
        row_list[b], row_count[b], row_full[b] = _lists(cls[b])
        col_list[b], col_count[b], col_full[b] = _lists(cls[b].T)
    return {
        "B": B, "L": L, "Lk": Lk, "block_m": block_m, "block_n": block_n, "nTq": nTq, "nTk": nTk,
        "q_nv": q_nv, "q_lo": q_lo, "q_hi": q_hi, "k_nv": k_nv, "k_lo": k_lo, "k_hi": k_hi,
        "cls": cls,
        "row_list": row_list, "row_count": row_count, "row_full": row_full,
        "col_list": col_list, "col_count": col_count, "col_full": col_full,
        "q_order": _longest_first(row_count.reshape(-1)),
        "k_order": _longest_first(col_count.reshape(-1)),
    }
