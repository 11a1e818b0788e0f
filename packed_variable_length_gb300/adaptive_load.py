"""Dual-constraint adaptive bucketing ("AdaptiveLoad" §2.A).

Equal-token bucketing caps a bucket's batch at B x S <= M_mem, so the batch
of a long-sequence bucket costs far more than that of a short one: attention
grows as S^2.  AdaptiveLoad adds a compute constraint B x S^p <= M_comp and
takes, per bucket shape S (tokens per sequence),

    B_shape = max(1, min(floor(M_mem / S), floor(M_comp / S^p))).

p and M_comp come from a cost model fitted to measured step times ("Shape
Benchmarking"): step_time ~ a + b B S^p, fitted by nonlinear least squares
over (a, b, p).  Here the fit is a variable projection: for a fixed p the
model is linear in (a, b) and solved exactly; the residual is then minimised
over p by a coarse scan and a golden-section refinement.

Readings (the page leaves these open):
- M_comp is the modelled cost of a memory-bound batch at a reference length
  S_ref: M_comp = floor(M_mem / S_ref) * S_ref^p.  Buckets shorter than S_ref
  are limited by memory and longer ones by compute.  The default S_ref is
  the shortest bucket, which makes every bucket's modelled cost about equal.
- Episodes are bucketed by their padded frame count (the pad-collate rule
  of "lingbot_va_packing" §2.1: F rounded up to a multiple of 8 latent
  frames), so S = tokens_per_frame * F_pad.
- A bucket's last, partial batch is kept: every episode is used once an epoch.
- Batches, not episodes, are dealt to the ranks round-robin (their sizes
  differ), after a seeded shuffle of the batch order.

Host-side logic only: the timings it is fitted to come from the library's
kernels (see bench.py's adaptive_load workload).
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np


def batch_size(S: float, m_mem: float, m_comp: float, p: float) -> int:
    """B_shape = max(1, min(floor(M_mem / S), floor(M_comp / S^p)))."""
    if S <= 0 or m_mem <= 0 or m_comp <= 0:
        raise ValueError("S, M_mem and M_comp must be positive")
    by_mem = math.floor(m_mem / S)
    by_comp = math.floor(m_comp / S ** p) if math.isfinite(m_comp) else by_mem
    return max(1, min(by_mem, by_comp))


def m_comp_for(m_mem: float, s_ref: float, p: float) -> float:
    """The compute bound that equals the modelled load of a memory-bound batch
    at length s_ref: floor(M_mem / s_ref) * s_ref^p."""
    if s_ref <= 0 or m_mem < s_ref:
        raise ValueError("need 0 < s_ref <= M_mem")
    return math.floor(m_mem / s_ref) * s_ref ** p


@dataclasses.dataclass
class CostModel:
    """step_time ~ a + b * B * S^p, with the fit's residual statistics."""
    a: float
    b: float
    p: float
    rss: float
    r2: float

    def predict(self, B, S):
        return self.a + self.b * np.asarray(B, dtype=np.float64) * np.asarray(S, dtype=np.float64) ** self.p


def _linear_fit(x: np.ndarray, t: np.ndarray):
    """Least squares t ~ a + b x; returns (a, b, rss)."""
    n = len(t)
    xm, tm = x.mean(), t.mean()
    dx = x - xm
    sxx = float(dx @ dx)
    if sxx == 0.0:
        return float(tm), 0.0, float(((t - tm) ** 2).sum())
    b = float(dx @ (t - tm)) / sxx
    a = float(tm - b * xm)
    r = t - a - b * x
    return a, b, float(r @ r) if n else 0.0


def fit_cost_model(B, S, t, p_lo: float = 0.5, p_hi: float = 3.0, scan: int = 251) -> CostModel:
    """Fits step_time ~ a + b B S^p to measured (B, S, t) by least squares.

    For each p the best (a, b) is exact (linear least squares on x = B S^p);
    the residual sum over p is scanned on `scan` points of [p_lo, p_hi] and
    the best bracket refined by golden-section search to ~1e-10."""
    B = np.asarray(B, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)
    if not (B.shape == S.shape == t.shape) or B.ndim != 1 or len(t) < 3:
        raise ValueError("need three or more (B, S, t) samples of equal length")
    if len(np.unique(S)) < 2:
        raise ValueError("the exponent needs two or more sequence lengths")
    s_scale = S.max()

    def rss(p):
        # S / s_scale keeps x well conditioned; b is rescaled at the end
        return _linear_fit(B * (S / s_scale) ** p, t)[2]

    grid = np.linspace(p_lo, p_hi, scan)
    vals = np.array([rss(p) for p in grid])
    i = int(np.argmin(vals))
    lo, hi = grid[max(i - 1, 0)], grid[min(i + 1, scan - 1)]
    g = (math.sqrt(5.0) - 1.0) / 2.0
    x1, x2 = hi - g * (hi - lo), lo + g * (hi - lo)
    f1, f2 = rss(x1), rss(x2)
    while hi - lo > 1e-10:
        if f1 <= f2:
            hi, x2, f2 = x2, x1, f1
            x1 = hi - g * (hi - lo)
            f1 = rss(x1)
        else:
            lo, x1, f1 = x1, x2, f2
            x2 = lo + g * (hi - lo)
            f2 = rss(x2)
    p = 0.5 * (lo + hi)
    if vals[i] < rss(p):  # an end point of the scan can beat the interior bracket
        p = float(grid[i])
    a, b_scaled, r = _linear_fit(B * (S / s_scale) ** p, t)
    tot = float(((t - t.mean()) ** 2).sum())
    return CostModel(a=a, b=b_scaled / s_scale ** p, p=float(p), rss=r, r2=1.0 - r / tot if tot > 0 else 1.0)


def padded_frames(F, pad_multiple: int):
    F = np.asarray(F, dtype=np.int64)
    return -(-F // pad_multiple) * pad_multiple


class DualConstraintBatchSampler:
    """Yields lists of episode indices, one list per batch, for one rank.

    lengths: latent frame counts F per episode.  Episodes are bucketed by
    F_pad = round_up(F, pad_multiple); a bucket of sequence length
    S = tokens_per_frame * F_pad takes batches of batch_size(S, m_mem,
    m_comp, p).  Each epoch (seed + epoch): shuffle the episodes, keep
    buckets in shuffled order, cut each into batches (last one partial),
    shuffle the batch order, deal batches to ranks round-robin.  With m_comp
    = inf this is equal-token bucketing (B = floor(M_mem / S))."""

    def __init__(self, lengths, tokens_per_frame: int, m_mem: float, m_comp: float = math.inf, p: float = 2.0,
                 pad_multiple: int = 8, rank: int = 0, world_size: int = 1, seed: int = 0):
        if tokens_per_frame <= 0 or pad_multiple <= 0 or world_size <= 0 or not (0 <= rank < world_size):
            raise ValueError("bad tokens_per_frame / pad_multiple / rank / world_size")
        self.lengths = np.asarray(lengths, dtype=np.int64)
        if (self.lengths <= 0).any():
            raise ValueError("episode lengths must be positive")
        self.T = int(tokens_per_frame)
        self.m_mem = float(m_mem)
        self.m_comp = float(m_comp)
        self.p = float(p)
        self.pad_multiple = int(pad_multiple)
        self.rank = int(rank)
        self.world_size = int(world_size)
        self.seed = int(seed)
        self.epoch = 0
        self.f_pad = padded_frames(self.lengths, self.pad_multiple)
        if (self.T * self.f_pad > self.m_mem).any():
            raise ValueError("an episode is longer than the memory bound M_mem")

    def set_epoch(self, epoch: int) -> None:
        self.epoch = int(epoch)

    def shape_batch_size(self, f_pad: int) -> int:
        return batch_size(self.T * int(f_pad), self.m_mem, self.m_comp, self.p)

    def all_batches(self) -> list[list[int]]:
        """Every rank's batches of this epoch, in dealing order."""
        rng = np.random.default_rng(self.seed + self.epoch)
        order = rng.permutation(len(self.lengths))
        out: list[list[int]] = []
        for fp in np.unique(self.f_pad):
            members = [int(i) for i in order if self.f_pad[i] == fp]
            bs = self.shape_batch_size(int(fp))
            out.extend(members[k:k + bs] for k in range(0, len(members), bs))
        perm = rng.permutation(len(out))
        return [out[i] for i in perm]

    def batches(self) -> list[list[int]]:
        return self.all_batches()[self.rank::self.world_size]

    def __iter__(self):
        return iter(self.batches())

    def __len__(self) -> int:
        return len(self.batches())


def coefficient_of_variation(x) -> float:
    """Population std / mean: the page's imbalance and sync-overhead measure."""
    x = np.asarray(x, dtype=np.float64)
    return float(x.std() / x.mean()) if len(x) and x.mean() != 0 else 0.0


def simulate_data_parallel(times, tokens, n_ranks: int):
    """Synchronous data parallelism over batches dealt round-robin: step k runs
    batches k*n .. k*n + n - 1 on n ranks and lasts as long as the slowest.
    Returns (tokens per second, per-step times, mean idle fraction of the ranks)."""
    times = np.asarray(times, dtype=np.float64)
    tokens = np.asarray(tokens, dtype=np.float64)
    n_steps = len(times) // n_ranks
    if n_steps == 0:
        raise ValueError("fewer batches than ranks")
    t = times[: n_steps * n_ranks].reshape(n_steps, n_ranks)
    step = t.max(axis=1)
    idle = float(((step[:, None] - t).sum() / (step.sum() * n_ranks)))
    return float(tokens[: n_steps * n_ranks].sum() / step.sum()), step, idle
