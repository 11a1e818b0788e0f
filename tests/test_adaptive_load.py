"""The AdaptiveLoad host logic (packed_variable_length_gb300.adaptive_load)
against the oracle (CPU): batch sizes bit for bit, the cost-model fit at least
as good as the oracle's brute force, the sampler's buckets and batches, the
balance measures; and a two-rank gloo run that deals the batches."""

import math
import os

import numpy as np
import pytest

import oracle.adaptive_load as ref
from packed_variable_length_gb300 import adaptive_load as al


def test_batch_size_matches_oracle():
    rng = np.random.default_rng(11)
    for _ in range(3000):
        S = int(rng.integers(1, 70000))
        m_mem = float(rng.choice([65536, 32768, 131072]))
        p = float(rng.uniform(0.8, 2.5))
        s_ref = float(rng.integers(1000, 20000))
        m_comp = float(rng.choice([math.inf, m_mem * s_ref ** (p - 1), float(rng.uniform(1e3, 1e12))]))
        assert al.batch_size(S, m_mem, m_comp, p) == ref.batch_size(S, m_mem, m_comp, p)


def test_m_comp_reading():
    # with the default reference (the shortest bucket) every longer bucket is compute bound
    p = 1.8
    s_ref = 3952
    m_comp = al.m_comp_for(65536, s_ref, p)
    assert m_comp == 16 * s_ref ** p
    assert al.batch_size(s_ref, 65536, m_comp, p) == 16
    for S in (5472, 7296, 13680):
        assert al.batch_size(S, 65536, m_comp, p) == max(1, math.floor(m_comp / S ** p))
    with pytest.raises(ValueError):
        al.m_comp_for(100, 200, 2.0)


@pytest.mark.parametrize("a,b,p,noise,seed", [(2e-3, 3e-11, 1.7, 0.0, 0), (1e-3, 5e-11, 1.6, 0.05, 3),
                                              (4e-4, 2e-9, 1.2, 0.02, 7), (0.0, 1e-12, 2.0, 0.0, 1)])
def test_fit_matches_oracle(a, b, p, noise, seed):
    rng = np.random.default_rng(seed)
    Bs, Ss = np.meshgrid([1, 2, 3, 4, 8], [3952, 5472, 7296, 9728, 11856, 13680])
    Bs, Ss = Bs.ravel().astype(float), Ss.ravel().astype(float)
    t = a + b * Bs * Ss ** p
    if noise:
        t = t * (1 + noise * rng.standard_normal(t.shape))
    m = al.fit_cost_model(Bs, Ss, t)
    ra, rb, rp, rrss = ref.fit_cost_model(Bs, Ss, t)
    assert abs(m.p - rp) <= 2e-5
    assert m.rss <= rrss * (1 + 1e-9) + 1e-30     # the refined optimum is no worse than the grid's
    np.testing.assert_allclose(m.predict(Bs, Ss), ra + rb * Bs * Ss ** rp, rtol=1e-3, atol=1e-9)
    if not noise:
        assert abs(m.p - p) <= 1e-6 and m.r2 > 1 - 1e-12


def test_fit_rejects_unidentifiable_input():
    with pytest.raises(ValueError):
        al.fit_cost_model([1, 2, 4], [4000, 4000, 4000], [1.0, 2.0, 4.0])
    with pytest.raises(ValueError):
        al.fit_cost_model([1, 2], [4000, 5000], [1.0, 2.0])


def _lengths(seed=1005, n=160):
    return np.random.default_rng(seed).integers(103, 363, size=n)


@pytest.mark.parametrize("m_comp_kind", ["equal_token", "dual"])
def test_sampler_buckets_match_oracle(m_comp_kind):
    F = _lengths()
    p = 1.9
    m_comp = math.inf if m_comp_kind == "equal_token" else al.m_comp_for(65536, 38 * 104, p)
    s = al.DualConstraintBatchSampler(F, 38, 65536, m_comp, p, pad_multiple=8, seed=7)
    batches = s.all_batches()
    used = sorted(i for b in batches for i in b)
    assert used == list(range(len(F)))                       # every episode once an epoch
    f_pad = al.padded_frames(F, 8)
    got = {}
    for b in batches:
        fp = {int(f_pad[i]) for i in b}
        assert len(fp) == 1                                   # one padded shape per batch
        got.setdefault(fp.pop(), []).append(len(b))
    want = ref.bucket_batch_sizes(F, 38, 8, 65536, m_comp, p)
    assert {k: sorted(v) for k, v in got.items()} == {k: sorted(v) for k, v in want.items()}
    for b in batches:                                         # both constraints hold for full batches
        S = 38 * int(f_pad[b[0]])
        assert len(b) * S <= 65536 or len(b) == 1
        if m_comp_kind == "dual":
            assert len(b) * S ** p <= m_comp or len(b) == 1


def test_sampler_epochs_and_ranks():
    F = _lengths()
    s0 = al.DualConstraintBatchSampler(F, 38, 65536, al.m_comp_for(65536, 3952, 2.0), 2.0, rank=0, world_size=2, seed=3)
    s1 = al.DualConstraintBatchSampler(F, 38, 65536, al.m_comp_for(65536, 3952, 2.0), 2.0, rank=1, world_size=2, seed=3)
    allb = s0.all_batches()
    assert s0.batches() == allb[0::2] and s1.batches() == allb[1::2]
    assert s0.all_batches() == allb                          # deterministic per epoch
    s0.set_epoch(1)
    assert s0.all_batches() != allb
    with pytest.raises(ValueError):
        al.DualConstraintBatchSampler([2000], 38, 65536)     # longer than M_mem


def test_balance_measures_match_oracle():
    rng = np.random.default_rng(2)
    times = rng.uniform(0.5, 3.0, size=37)
    tokens = rng.integers(1000, 60000, size=37)
    assert abs(al.coefficient_of_variation(times) - ref.coefficient_of_variation(times)) < 1e-12
    for n in (1, 2, 8):
        tps, step, idle = al.simulate_data_parallel(times, tokens, n)
        assert abs(tps - ref.data_parallel_throughput(list(times), list(tokens), n)) <= 1e-9 * tps
        assert 0.0 <= idle < 1.0 and len(step) == len(times) // n


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    F = _lengths()
    s = al.DualConstraintBatchSampler(F, 38, 65536, al.m_comp_for(65536, 3952, 1.8), 1.8,
                                      rank=rank, world_size=world, seed=9)
    mine = s.batches()
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    if rank == 0:
        out.put(gathered)
    dist.destroy_process_group()


def test_two_gloo_ranks_partition_the_epoch():
    """Each rank builds its own share; together they cover every episode once."""
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    gathered = q.get(timeout=120)
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    episodes = sorted(i for share in gathered for b in share for i in b)
    assert episodes == list(range(160))
    assert abs(len(gathered[0]) - len(gathered[1])) <= 1
