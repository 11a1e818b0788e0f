"""Oracle: AdaptiveLoad's dual-constraint batch size, its cost-model fit and
the load-balance measures, in plain fp64.  TEST INFRASTRUCTURE ONLY (see the
package docstring).

"AdaptiveLoad" §2.A: a bucket of sequence length S gets the batch size

    B_shape = max(1, min(floor(M_mem / S), floor(M_comp / S^p)))

(memory constraint B S <= M_mem, compute constraint B S^p <= M_comp), and p,
M_comp come from the cost model step_time ~ a + b B S^p fitted to measured
step times by nonlinear least squares.  §4 measures load imbalance as the
coefficient of variation of the compute load and the synchronisation
overhead as the coefficient of variation of the step time.

The fit here is the least-squares definition evaluated by brute force: for
every p on a grid of spacing 1e-5 the best (a, b) solves the 2 x 2 normal
equations exactly, and the grid point of least residual is returned.
"""

from __future__ import annotations

import math

import numpy as np


def batch_size(S, m_mem, m_comp, p) -> int:
    # floor(min(x, y)) = min(floor(x), floor(y)); an infinite M_comp leaves the memory bound
    return max(1, math.floor(min(m_mem / S, m_comp / S ** p)))


def fit_cost_model(B, S, t, p_lo: float = 0.5, p_hi: float = 3.0, step: float = 1e-5):
    """Returns (a, b, p, rss) minimising sum (t - a - b B S^p)^2 with p on the grid."""
    B = np.asarray(B, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)
    n = len(t)
    best = None
    ps = np.arange(p_lo, p_hi + step / 2, step)
    for c0 in range(0, len(ps), 4096):
        pc = ps[c0:c0 + 4096]
        x = B[None, :] * S[None, :] ** pc[:, None]          # [grid, n]
        sx, sxx = x.sum(axis=1), (x * x).sum(axis=1)
        st, sxt = t.sum(), (x * t[None, :]).sum(axis=1)
        det = n * sxx - sx * sx
        b = (n * sxt - sx * st) / det
        a = (st - b * sx) / n
        r = t[None, :] - a[:, None] - b[:, None] * x
        rss = (r * r).sum(axis=1)
        k = int(np.argmin(rss))
        if best is None or rss[k] < best[3]:
            best = (float(a[k]), float(b[k]), float(pc[k]), float(rss[k]))
    return best


def bucket_batch_sizes(lengths, tokens_per_frame, pad_multiple, m_mem, m_comp, p):
    """{F_pad: [batch sizes]} of one epoch: each bucket of n episodes cut into
    batches of B_shape, the last one holding the remainder."""
    lengths = np.asarray(lengths, dtype=np.int64)
    f_pad = ((lengths + pad_multiple - 1) // pad_multiple) * pad_multiple
    out = {}
    for fp in sorted(set(int(v) for v in f_pad)):
        n = int((f_pad == fp).sum())
        bs = batch_size(tokens_per_frame * fp, m_mem, m_comp, p)
        sizes = [bs] * (n // bs) + ([n % bs] if n % bs else [])
        out[fp] = sizes
    return out


def coefficient_of_variation(x) -> float:
    x = np.asarray(x, dtype=np.float64)
    mean = x.sum() / len(x)
    return float(math.sqrt(((x - mean) ** 2).sum() / len(x)) / mean)


def data_parallel_throughput(times, tokens, n_ranks):
    """Steps of n_ranks consecutive batches, each as long as its slowest batch:
    tokens per second over the whole steps (a trailing partial step is dropped)."""
    n_steps = len(times) // n_ranks
    total_t = 0.0
    total_tok = 0.0
    for k in range(n_steps):
        total_t += max(times[k * n_ranks:(k + 1) * n_ranks])
        total_tok += sum(tokens[k * n_ranks:(k + 1) * n_ranks])
    return total_tok / total_t
