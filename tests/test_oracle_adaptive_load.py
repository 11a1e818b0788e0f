"""The AdaptiveLoad oracle against independent checks (CPU only): hand-worked
batch sizes and the formula's limiting cases, recovery of known cost models,
optimality against numpy's own least squares and scipy's curve_fit, brute
force on the bucket split, closed forms of the balance measures, and planted
mistakes that the checks must catch."""

import math
import os
import types

import numpy as np
import pytest

import oracle.adaptive_load as al

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "adaptive_load.py")


def check_batch_size_table(mod):
    m_mem = 65536
    m_comp = 65536 * 3952.0          # the cost of a full batch at S = 3952 with p = 2
    # S = 3952 (104 frames x 38): memory and compute both allow 16
    assert mod.batch_size(3952, m_mem, m_comp, 2.0) == 16
    # S = 13680 (360 frames x 38): memory 4, compute floor(1.386) = 1
    assert mod.batch_size(13680, m_mem, m_comp, 2.0) == 1
    # S = 6080 (160 frames): memory floor(10.78) = 10, compute floor(7.006) = 7
    assert mod.batch_size(6080, m_mem, m_comp, 2.0) == 7
    # a sequence longer than the memory bound still gets a batch of one
    assert mod.batch_size(70000, m_mem, m_comp, 2.0) == 1
    # p = 1 with M_comp = M_mem is equal-token bucketing
    for S in (100, 3952, 6080, 13680, 65536):
        assert mod.batch_size(S, m_mem, m_mem, 1.0) == m_mem // S
    # an unbounded compute budget leaves the memory bound alone
    assert mod.batch_size(6080, m_mem, math.inf, 2.0) == 10
    # a compute bound that binds exactly: 4 x 100^1.5 = 4000
    assert mod.batch_size(100, 10 ** 6, 4000.0, 1.5) == 4


def _samples(a, b, p, noise=0.0, seed=0):
    rng = np.random.default_rng(seed)
    Bs, Ss = np.meshgrid([1, 2, 4, 8], [3952, 5472, 7296, 9728, 13680])
    Bs, Ss = Bs.ravel().astype(float), Ss.ravel().astype(float)
    t = a + b * Bs * Ss ** p
    if noise:
        t = t * (1 + noise * rng.standard_normal(t.shape))
    return Bs, Ss, t


def check_fit_recovers_known_models(mod):
    for a, b, p in ((2e-3, 3e-11, 1.7), (5e-4, 1e-9, 1.25), (0.0, 2e-12, 2.0), (1e-2, 4e-10, 1.5)):
        Bs, Ss, t = _samples(a, b, p)
        fa, fb, fp, rss = mod.fit_cost_model(Bs, Ss, t)
        assert abs(fp - p) <= 1e-5, (p, fp)
        assert rss <= 1e-6 * float((t ** 2).sum())
        pred = fa + fb * Bs * Ss ** fp
        assert np.abs(pred - t).max() <= 1e-4 * t.max()


def check_fit_is_least_squares(mod):
    """On noisy data the returned (a, b) are numpy's least squares at that p,
    no other p near it does better, and scipy's curve_fit lands there too."""
    Bs, Ss, t = _samples(1e-3, 5e-11, 1.6, noise=0.05, seed=3)
    fa, fb, fp, rss = mod.fit_cost_model(Bs, Ss, t)
    X = np.stack([np.ones_like(Bs), Bs * Ss ** fp], axis=1)
    coef, *_ = np.linalg.lstsq(X, t, rcond=None)
    assert abs(coef[0] - fa) <= 1e-9 + 1e-6 * abs(fa) and abs(coef[1] - fb) <= 1e-6 * abs(fb)
    for dp in (-1e-2, -1e-3, 1e-3, 1e-2):
        Xd = np.stack([np.ones_like(Bs), Bs * Ss ** (fp + dp)], axis=1)
        cd, *_ = np.linalg.lstsq(Xd, t, rcond=None)
        assert ((t - Xd @ cd) ** 2).sum() >= rss * (1 - 1e-9)
    scipy_opt = pytest.importorskip("scipy.optimize")
    popt, _ = scipy_opt.curve_fit(lambda x, a, b, p: a + b * x[0] * x[1] ** p, (Bs, Ss), t,
                                  p0=(fa * 1.1, fb * 0.9, fp + 0.05), maxfev=20000)
    assert abs(popt[2] - fp) <= 1e-3


def check_bucket_split(mod):
    rng = np.random.default_rng(5)
    F = rng.integers(103, 363, size=160)
    sizes = mod.bucket_batch_sizes(F, 38, 8, 65536, 65536 * 3952.0, 2.0)
    f_pad = ((F + 7) // 8) * 8
    for fp, bs in sizes.items():
        n = int((f_pad == fp).sum())
        assert sum(bs) == n
        full = mod.batch_size(38 * fp, 65536, 65536 * 3952.0, 2.0)
        assert all(s == full for s in bs[:-1]) and 0 < bs[-1] <= full
    assert sorted(sizes) == sorted(set(int(v) for v in f_pad))
    # a hand case: 5 episodes of 104 frames at 16 per batch -> one batch of 5
    assert mod.bucket_batch_sizes([100] * 5, 38, 8, 65536, 65536 * 3952.0, 2.0) == {104: [5]}


def check_balance_measures(mod):
    assert mod.coefficient_of_variation([2.0, 2.0, 2.0]) == 0.0
    assert abs(mod.coefficient_of_variation([1.0, 3.0]) - 0.5) < 1e-15
    # two ranks: steps (1, 3) and (2, 2) last 3 and 2; 10 tokens each batch
    assert abs(mod.data_parallel_throughput([1.0, 3.0, 2.0, 2.0], [10] * 4, 2) - 40 / 5) < 1e-12
    # a trailing partial step is dropped
    assert abs(mod.data_parallel_throughput([1.0, 3.0, 2.0], [10] * 3, 2) - 20 / 3) < 1e-12


CHECKS = [check_batch_size_table, check_fit_recovers_known_models, check_fit_is_least_squares,
          check_bucket_split, check_balance_measures]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_check(check):
    check(al)


MUTATIONS = {
    "ceil_not_floor": ("return max(1, math.floor(min(m_mem / S, m_comp / S ** p)))",
                       "return max(1, math.ceil(min(m_mem / S, m_comp / S ** p)))"),
    "max_not_min": ("return max(1, math.floor(min(m_mem / S, m_comp / S ** p)))",
                    "return max(1, math.floor(max(m_mem / S, m_comp / S ** p)))"),
    "linear_not_power": ("return max(1, math.floor(min(m_mem / S, m_comp / S ** p)))",
                         "return max(1, math.floor(min(m_mem / S, m_comp / (S * p))))"),
    "no_floor_of_one": ("return max(1, math.floor(min(m_mem / S, m_comp / S ** p)))",
                        "return math.floor(min(m_mem / S, m_comp / S ** p))"),
    "fit_without_intercept": ("        a = (st - b * sx) / n\n", "        a = 0.0 * sx\n"),
    "fit_linear_in_s": ("x = B[None, :] * S[None, :] ** pc[:, None]", "x = B[None, :] * S[None, :] * pc[:, None]"),
    "remainder_dropped": ("sizes = [bs] * (n // bs) + ([n % bs] if n % bs else [])", "sizes = [bs] * (n // bs)"),
    "cv_sample_std": ("return float(math.sqrt(((x - mean) ** 2).sum() / len(x)) / mean)",
                      "return float(math.sqrt(((x - mean) ** 2).sum() / (len(x) - 1)) / mean)"),
    "dp_mean_not_max": ("total_t += max(times[k * n_ranks:(k + 1) * n_ranks])",
                        "total_t += sum(times[k * n_ranks:(k + 1) * n_ranks]) / n_ranks"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_checks_catch_mutant(name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType("adaptive_load_mutant")
    exec(compile(src.replace(old, new), "adaptive_load_mutant", "exec"), mod.__dict__)
    caught = []
    for check in CHECKS:
        try:
            check(mod)
        except (AssertionError, ValueError, IndexError, ZeroDivisionError, OverflowError):
            caught.append(check.__name__)
    assert caught, f"no check caught {name}"
