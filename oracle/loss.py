"""Oracle: the frame_valid-masked mean-squared-error loss and its gradient,
fp64 on the CPU.  TEST INFRASTRUCTURE ONLY (see the package docstring).

"lingbot_va_packing" §2.1 (compute_loss) and "furniture_packing_variable_length"
(the loss paragraph): the collate function returns each episode's number of
real latent frames, valid_frames[b]; compute_loss builds

    frame_valid[b, f] = f < valid_frames[b]        (f = 0 .. F-1)

and averages the latent and the action losses over the valid frames only, so
padding frames take no part in the loss or its gradient.  Per stream, with
tokens laid out frame-major (token n of row b belongs to frame n // T, T
tokens per frame) and C values per token:

    valid[b, n] = frame_valid[b, n // T]
    loss        = sum_{b, n : valid} sum_c (pred - target)^2 / (C * n_valid)
    dloss/dpred = 2 (pred - target) / (C * n_valid) on valid tokens, 0 elsewhere

n_valid is the number of valid tokens (so the loss is the mean over valid
frames of each frame's mean squared error: every frame has T tokens).  A
batch with no valid token has loss 0 and gradient 0.

Readings (the pages name the mask and the averaging, not the per-element
loss): the per-element loss is the squared error of the prediction, the
flow-matching objective of the Wan-family models the pages train; the mean
pools all valid frames of the batch (not a mean of per-episode means).

``valid_from_seq_id`` gives the same token mask from the attention's seq_ids
(seq_id >= 0), which is how the mask reaches the loss on concatenated rows.
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


def frame_valid_tokens(valid_frames, F: int, T: int) -> np.ndarray:
    """Token mask [B, F*T] from the per-episode valid frame counts."""
    valid_frames = np.asarray(valid_frames, dtype=np.int64).reshape(-1)
    frame_valid = np.arange(F)[None, :] < valid_frames[:, None]   # [B, F]
    return np.repeat(frame_valid, T, axis=1)


def valid_from_seq_id(seq_id) -> np.ndarray:
    """Token mask [B, L]: the tokens the attention keeps (seq_id >= 0)."""
    return np.asarray(seq_id) >= 0


def _check(pred, target, valid):
    if len(pred.shape) != 3 or tuple(pred.shape) != tuple(target.shape):
        raise ValueError("pred and target must be [B, L, C] of the same shape")
    if tuple(np.asarray(valid).shape) != tuple(pred.shape[:2]):
        raise ValueError("valid must be [B, L]")


def masked_mse(pred, target, valid):
    """Returns (loss, n_valid): the mean of (pred - target)^2 over the valid
    tokens' elements; loss 0 when no token is valid."""
    _check(pred, target, valid)
    p, t = _f64(pred), _f64(target)
    valid = np.asarray(valid, dtype=bool)
    C = p.shape[2]
    n_valid = int(valid.sum())
    if n_valid == 0:
        return 0.0, 0
    diff = (p - t)[valid]                  # [n_valid, C]
    return float((diff * diff).sum() / (C * n_valid)), n_valid


def masked_mse_grad(pred, target, valid, dloss: float = 1.0):
    """Returns dloss * d loss / d pred [B, L, C] (zero on invalid tokens)."""
    _check(pred, target, valid)
    p, t = _f64(pred), _f64(target)
    valid = np.asarray(valid, dtype=bool)
    C = p.shape[2]
    n_valid = int(valid.sum())
    g = np.zeros_like(p)
    if n_valid == 0:
        return g
    g[valid] = (2.0 * float(dloss) / (C * n_valid)) * (p - t)[valid]
    return g
