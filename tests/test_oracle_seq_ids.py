"""seq_id oracle against closed forms, the pages' worked example and a
position-by-position restatement (CPU only)."""

import numpy as np
import pytest

import golden_io
import oracle
import workloads as wl


def per_position(seg_frames, seg_valid, T, L):
    """For every position p: walk the segments to find its frame (separate code)."""
    B, K = seg_frames.shape
    out = np.empty((B, L), np.int64)
    for b in range(B):
        for p in range(L):
            frame = p // T
            sid = -1
            for k in range(K):
                if frame < seg_frames[b, k]:
                    sid = b * K + k if frame < seg_valid[b, k] else -1
                    break
                frame -= seg_frames[b, k]
            out[b, p] = sid
    return out


def test_pages_padded_batch_example():
    g = golden_io.load("padded_batch.txt")
    assert int(wl.round_up(max(g["valid_frames"]), g["pad_multiple"])) == g["padded_frames"]
    lay = wl.config_layout(3)
    assert lay.seg_valid[:, 0].tolist() == g["valid_frames"]
    assert (lay.seg_frames == g["padded_frames"]).all()
    sid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    for b, v in enumerate(g["valid_frames"]):
        n = v * lay.tokens_per_frame
        assert (sid[b, :n] == b).all() and (sid[b, n:] == -1).all()
    lay2 = wl.config_layout(2)
    assert (lay2.seg_frames == g["same_length_frames"]).all()


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_workload_closed_form(n):
    lay = wl.config_layout(n)
    sid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    T = lay.tokens_per_frame
    expect = np.full((lay.B, lay.L), -1)
    for b in range(lay.B):
        start = 0
        for k in range(lay.K):
            nvalid = lay.seg_valid[b, k] * T
            expect[b, start:start + nvalid] = b * lay.K + k
            start += lay.seg_frames[b, k] * T
    np.testing.assert_array_equal(sid, expect)


@pytest.mark.parametrize("seed", range(6))
def test_random_layouts_per_position(seed):
    rng = np.random.default_rng(seed)
    lay = wl.random_layout(rng, B=3, K=4, T=int(rng.integers(1, 7)), L=int(rng.integers(1, 300)),
                           H=1, D=8)
    sid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    np.testing.assert_array_equal(sid, per_position(lay.seg_frames, lay.seg_valid,
                                                    lay.tokens_per_frame, lay.L))


def test_rejects_bad_tables():
    with pytest.raises(ValueError):
        oracle.build_seq_ids([[5]], [[6]], 2, 100)      # valid > frames
    with pytest.raises(ValueError):
        oracle.build_seq_ids([[51]], [[1]], 2, 100)     # needs 102 > L tokens
    with pytest.raises(ValueError):
        oracle.build_seq_ids([[-1]], [[0]], 2, 100)     # negative
