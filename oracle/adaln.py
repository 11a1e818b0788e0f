"""Oracle: LayerNorm followed by AdaLN modulation, and its gradient, fp64 on
the CPU.  TEST INFRASTRUCTURE ONLY (see the package docstring).

"AdaptiveLoad" §2.B fuses the adaptive layer norm of a DiT / MMDiT block
(normalisation, then the modulation by the conditioning) into one kernel:
per token, mean and variance over the feature dimension D, then the linear
modulation on the way out; the backward reduces the modulation gradients
over the sequence dimension N.  Per batch row b, token n, feature d, with
the inputs exactly as handed to the kernels (bf16 x upcast to fp64, fp32
shift / scale upcast to fp64):

    mu_n    = (1/D) sum_d x_nd
    var_n   = (1/D) sum_d (x_nd - mu_n)^2
    r_n     = 1 / sqrt(var_n + eps)
    xh_nd   = (x_nd - mu_n) r_n
    y_nd    = xh_nd (1 + scale_bd) + shift_bd

and, for an upstream gradient dy,

    g_nd      = dy_nd (1 + scale_bd)
    dx_nd     = r_n (g_nd - mean_d(g_n) - xh_nd mean_d(g_n xh_n))
    dshift_bd = sum_n dy_nd
    dscale_bd = sum_n dy_nd xh_nd

Readings (the page gives no formulas): the layer norm has no elementwise
affine of its own (the modulation is the affine, as in DiT's adaptive layer
norm), eps = 1e-6 unless passed, and shift / scale are one vector per batch
row shared by all its tokens.  The variance is the biased (1/D) one.
"""

from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _check(x, shift, scale):
    if len(x.shape) != 3:
        raise ValueError("x must be [B, N, D]")
    B, _, D = x.shape
    if tuple(shift.shape) != (B, D) or tuple(scale.shape) != (B, D):
        raise ValueError("shift and scale must be [B, D]")


def adaln_fwd(x, shift, scale, eps: float = 1e-6):
    """Returns (y [B, N, D], mean [B, N], rstd [B, N]) in fp64."""
    _check(x, shift, scale)
    x, shift, scale = _f64(x), _f64(shift), _f64(scale)
    mu = x.mean(axis=2)
    xc = x - mu[:, :, None]
    var = (xc * xc).mean(axis=2)
    r = 1.0 / np.sqrt(var + eps)
    xh = xc * r[:, :, None]
    y = xh * (1.0 + scale[:, None, :]) + shift[:, None, :]
    return y, mu, r


def adaln_bwd(x, shift, scale, dy, eps: float = 1e-6):
    """Returns (dx [B, N, D], dshift [B, D], dscale [B, D]) in fp64.  The row
    statistics are recomputed from x; nothing produced by a kernel enters."""
    _check(x, shift, scale)
    x, scale, dy = _f64(x), _f64(scale), _f64(dy)
    D = x.shape[2]
    mu = x.mean(axis=2)
    xc = x - mu[:, :, None]
    r = 1.0 / np.sqrt((xc * xc).mean(axis=2) + eps)
    xh = xc * r[:, :, None]
    g = dy * (1.0 + scale[:, None, :])
    mg = g.sum(axis=2) / D
    mgx = (g * xh).sum(axis=2) / D
    dx = r[:, :, None] * (g - mg[:, :, None] - xh * mgx[:, :, None])
    dshift = dy.sum(axis=1)
    dscale = (dy * xh).sum(axis=1)
    return dx, dshift, dscale
