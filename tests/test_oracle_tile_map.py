"""Tile-map oracle against brute-force pair enumeration and closed forms (CPU)."""

import numpy as np
import pytest

import oracle
import workloads as wl
from oracle import EMPTY, FULL, PARTIAL


def admissible(sid_row, L, bm, bn, qt, kt):
    """Matrix of admissible pairs of one tile pair, by enumeration."""
    qs = [p for p in range(qt * bm, (qt + 1) * bm)]
    ks = [p for p in range(kt * bn, (kt + 1) * bn)]
    m = np.zeros((bm, bn), bool)
    for a, i in enumerate(qs):
        for c, j in enumerate(ks):
            if i < L and j < L and sid_row[i] >= 0 and sid_row[i] == sid_row[j]:
                m[a, c] = True
    return m


def check_sound(sid, L, bm, bn, exact):
    tm = oracle.build_tile_map(sid, L, bm, bn)
    for b in range(sid.shape[0]):
        for qt in range(tm["nTq"]):
            for kt in range(tm["nTk"]):
                m = admissible(sid[b], L, bm, bn, qt, kt)
                c = tm["cls"][b, qt, kt]
                if c == EMPTY:
                    assert not m.any()
                if c == FULL:
                    assert m.all()
                if m.all():  # every pair admissible: both tiles whole and valid
                    assert c == FULL
                if exact:
                    assert (c == EMPTY) == (not m.any())
    return tm


def check_lists(tm):
    B, nTq, nTk = tm["cls"].shape
    for b in range(B):
        for name, cls, lst, cnt, nfull in (("row", tm["cls"][b], tm["row_list"][b], tm["row_count"][b], tm["row_full"][b]),
                                           ("col", tm["cls"][b].T, tm["col_list"][b], tm["col_count"][b], tm["col_full"][b])):
            for i in range(cls.shape[0]):
                full = [j for j in range(cls.shape[1]) if cls[i, j] == FULL]
                part = [j for j in range(cls.shape[1]) if cls[i, j] == PARTIAL]
                assert cnt[i] == len(full) + len(part) and nfull[i] == len(full), name
                assert list(lst[i, :cnt[i]]) == full + part, name
                assert (lst[i, cnt[i]:] == -1).all(), name
    for key, cnt in (("q_order", tm["row_count"]), ("k_order", tm["col_count"])):
        flat = cnt.reshape(-1)
        order = tm[key]
        assert sorted(order.tolist()) == list(range(len(flat)))
        for a, c in zip(order[:-1], order[1:]):
            assert flat[a] > flat[c] or (flat[a] == flat[c] and a < c)


@pytest.mark.parametrize("seed", range(5))
def test_monotone_layouts_exact(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(20, 90))
    lay = wl.random_layout(rng, B=2, K=3, T=int(rng.integers(1, 5)), L=L, H=1, D=8)
    sid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, L)
    bm, bn = [(8, 8), (8, 16), (16, 8)][seed % 3]
    tm = check_sound(sid, L, bm, bn, exact=True)
    check_lists(tm)
    if bm == bn:
        np.testing.assert_array_equal(tm["cls"], tm["cls"].transpose(0, 2, 1))


@pytest.mark.parametrize("seed", range(4))
def test_interleaved_ids_sound(seed):
    rng = np.random.default_rng(100 + seed)
    L = int(rng.integers(10, 70))
    sid = rng.integers(-1, 4, size=(2, L)).astype(np.int32)
    tm = check_sound(sid, L, 8, 8, exact=False)
    check_lists(tm)


@pytest.mark.parametrize("n", [2, 3, 4])
def test_workload_class_counts(n):
    """One id per contiguous run: per row/episode with n_e valid tokens starting
    on a tile boundary, f = n_e // 128 whole tiles are FULL with each other."""
    lay = wl.config_layout(n)
    sid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    tm = oracle.build_tile_map(sid, lay.L, 128, 128)
    nT = -(-lay.L // 128)
    if n in (2, 3):
        for b in range(lay.B):
            nval = int(lay.seg_valid[b, 0]) * lay.tokens_per_frame
            f, r = divmod(nval, 128)
            assert (tm["cls"][b] == FULL).sum() == f * f
            assert (tm["cls"][b] == PARTIAL).sum() == (2 * f + 1 if r else 0)
            assert (tm["cls"][b] != EMPTY).sum() == (f + (1 if r else 0)) ** 2
            assert tm["cls"][b].shape == (nT, nT)
    else:
        check_sound_blocks = (tm["cls"][0] != EMPTY)
        # non-empty iff the tiles share an episode (monotone layout)
        starts = np.concatenate([[0], np.cumsum(lay.seg_frames[0]) * lay.tokens_per_frame])
        for qt in range(nT):
            for kt in range(nT):
                eq = set(range(len(starts) - 1))
                q_eps = {e for e in eq if starts[e] < min((qt + 1) * 128, lay.L) and starts[e + 1] > qt * 128}
                k_eps = {e for e in eq if starts[e] < min((kt + 1) * 128, lay.L) and starts[e + 1] > kt * 128}
                assert check_sound_blocks[qt, kt] == bool(q_eps & k_eps)


# ---------------------------------------------------------- cross attention
def admissible_cross(qsid_row, ksid_row, Lq, Lk, bm, bn, qt, kt):
    m = np.zeros((bm, bn), bool)
    for a in range(bm):
        for c in range(bn):
            i, j = qt * bm + a, kt * bn + c
            if i < Lq and j < Lk and qsid_row[i] >= 0 and qsid_row[i] == ksid_row[j]:
                m[a, c] = True
    return m


def check_sound_cross(qsid, ksid, Lq, Lk, bm, bn, exact):
    tm = oracle.build_tile_map(qsid, Lq, bm, bn, k_seq_id=ksid, Lk=Lk)
    assert tm["cls"].shape == (qsid.shape[0], -(-Lq // bm), -(-Lk // bn))
    for b in range(qsid.shape[0]):
        for qt in range(tm["nTq"]):
            for kt in range(tm["nTk"]):
                m = admissible_cross(qsid[b], ksid[b], Lq, Lk, bm, bn, qt, kt)
                c = tm["cls"][b, qt, kt]
                if c == EMPTY:
                    assert not m.any()
                if c == FULL:
                    assert m.all()
                if m.all():
                    assert c == FULL
                if exact:
                    assert (c == EMPTY) == (not m.any())
    return tm


@pytest.mark.parametrize("seed", range(4))
def test_cross_monotone_layouts_exact(seed):
    """Queries and keys of the same episodes laid out in the same order with
    different tokens per frame (the latent / action streams)."""
    rng = np.random.default_rng(200 + seed)
    lay = wl.random_layout(rng, B=2, K=3, T=int(rng.integers(2, 6)), L=int(rng.integers(40, 90)), H=1, D=8)
    Tk = int(rng.integers(1, 4))
    Lk = int(lay.seg_frames.sum(axis=1).max()) * Tk + int(rng.integers(0, 9))
    qsid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    ksid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, Tk, Lk)
    bm, bn = [(8, 8), (8, 4), (16, 8), (4, 8)][seed]
    tm = check_sound_cross(qsid, ksid, lay.L, Lk, bm, bn, exact=True)
    check_lists(tm)


@pytest.mark.parametrize("seed", range(3))
def test_cross_interleaved_ids_sound(seed):
    rng = np.random.default_rng(300 + seed)
    Lq, Lk = int(rng.integers(10, 60)), int(rng.integers(5, 40))
    qsid = rng.integers(-1, 4, size=(2, Lq)).astype(np.int32)
    ksid = rng.integers(-1, 5, size=(2, Lk)).astype(np.int32)
    tm = check_sound_cross(qsid, ksid, Lq, Lk, 8, 8, exact=False)
    check_lists(tm)


def test_cross_with_own_ids_is_self():
    rng = np.random.default_rng(7)
    sid = rng.integers(-1, 3, size=(2, 50)).astype(np.int32)
    a = oracle.build_tile_map(sid, 50, 8, 16)
    b = oracle.build_tile_map(sid, 50, 8, 16, k_seq_id=sid, Lk=50)
    for key in ("cls", "row_list", "col_list", "q_order", "k_order"):
        np.testing.assert_array_equal(a[key], b[key])
