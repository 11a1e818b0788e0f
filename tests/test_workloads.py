"""Input generators: shapes, seeding and the length-bucketing sampler (CPU)."""

import numpy as np
import torch

import golden_io
import workloads as wl


def test_sampler_pages_counts():
    g = golden_io.load("sampler_stats.txt")
    layouts, batches, lengths = wl.bucket_sweep_layouts()
    assert len(batches) == g["batches_per_epoch_per_rank"]
    assert all(len(b) == g["batch_size"] for b in batches)
    assert lengths.min() >= g["f_min"] and lengths.max() <= g["f_max"]
    assert sorted(i for b in batches for i in b) == list(range(len(lengths)))
    assert wl.padding_waste(batches, lengths, 8) < g["max_waste"]
    for lay, b in zip(layouts, batches):
        assert lay.L == int(wl.round_up(lengths[b].max(), 8)) * 38


def test_sampler_ranks_equal_batches_and_cover():
    lengths = np.arange(103, 103 + 37)
    shares = []
    for r in range(3):
        s = wl.LengthBucketBatchSampler(lengths, 4, r, 3, seed=7, pool_factor=2)
        shares.append(s.batches())
    assert len({len(s) for s in shares}) == 1
    seen = {i for s in shares for b in s for i in b}
    assert seen == set(range(len(lengths)))


def test_sampler_sorted_within_pool_and_epoch_changes():
    lengths = np.random.default_rng(0).integers(103, 363, 400)
    s = wl.LengthBucketBatchSampler(lengths, 4, 0, 1, seed=3, pool_factor=25)
    e0 = s.batches()
    s.set_epoch(1)
    e1 = s.batches()
    assert e0 != e1
    # within each pool of 100 episodes the batches are cut from sorted runs
    for b in e0:
        f = lengths[b]
        assert list(f) == sorted(f)


def test_tensors_seeded_and_bf16():
    lay = wl.config_layout(1)
    a = wl.make_tensors(lay)
    b = wl.make_tensors(lay)
    for k in ("q", "k", "v", "do"):
        assert a[k].dtype == torch.bfloat16 and a[k].shape == (2, 256, 2, 64)
        assert torch.equal(a[k], b[k])
    assert not torch.equal(a["q"], a["k"])


def test_concat64k_fits():
    lay = wl.config_layout(4)
    assert lay.K == 7 and lay.L == 65536
    assert int(lay.seg_frames.sum()) * 38 <= 65536
    assert (lay.seg_frames % 8 == 0).all()
    assert (lay.seg_frames >= 104).all() and (lay.seg_frames <= 368).all()


def test_random_layout_fits():
    rng = np.random.default_rng(5)
    for _ in range(50):
        L = int(rng.integers(1, 500))
        T = int(rng.integers(1, 40))
        lay = wl.random_layout(rng, 3, 5, T, L, 1, 8)
        assert (lay.seg_frames.sum(1) * T <= L).all()
        assert (lay.seg_valid <= lay.seg_frames).all() and (lay.seg_valid >= 0).all()
