"""torch.autograd wrapper: packed masked attention as a differentiable op.

The tile map is an explicit argument of both passes, so the backward always
sees the mask of its own forward (the class-attribute block-mask hazard of
"lingbot_va_packing" §2.2 cannot occur).
"""

from __future__ import annotations

import torch

from . import api


class _PackedAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, seq_id, k_seq_id, tile_map, scale):
        o, lse = api.masked_attn_fwd(q, k, v, seq_id, tile_map, scale, k_seq_id=k_seq_id)
        ctx.save_for_backward(q, k, v, o, lse, seq_id, k_seq_id)
        ctx.tile_map = tile_map
        ctx.scale = scale
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, seq_id, k_seq_id = ctx.saved_tensors
        dq, dk, dv = api.masked_attn_bwd(q, k, v, o, do.contiguous(), lse, seq_id, ctx.tile_map, ctx.scale,
                                         k_seq_id=k_seq_id)
        return dq, dk, dv, None, None, None, None


def packed_attention(q, k, v, seq_id, tile_map=None, scale=None, k_seq_id=None):
    """O = masked softmax attention of bf16 [B, L, H, D] q/k/v under int32 [B, L]
    seq_id; with k_seq_id (int32 [B, Lk]) cross attention of q [B, L, H, D]
    against k, v [B, Lk, H, D] ("lingbot_va_packing" §2.1)."""
    if tile_map is None:
        tile_map = api.tile_map_build(seq_id, k_seq_id=k_seq_id)
    return _PackedAttention.apply(q, k, v, seq_id, k_seq_id, tile_map, scale)


class _AdaLNModulate(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, shift, scale, eps):
        y = api.adaln_fwd(x, shift, scale, eps)
        ctx.save_for_backward(x, scale)
        ctx.eps = eps
        return y

    @staticmethod
    def backward(ctx, dy):
        x, scale = ctx.saved_tensors
        dx, dshift, dscale = api.adaln_bwd(x, scale, dy.contiguous(), ctx.eps)
        return dx, dshift, dscale, None


def adaln_modulate(x, shift, scale, eps: float = 1e-6):
    """layer_norm(x) * (1 + scale) + shift over bf16 x [B, N, D] with fp32
    shift / scale [B, D], differentiable ("AdaptiveLoad" §2.B); the backward
    recomputes the row statistics from x."""
    return _AdaLNModulate.apply(x, shift, scale, eps)


class _MaskedMSE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, pred, target, seq_id):
        loss = api.masked_mse_loss(pred, target, seq_id)
        ctx.save_for_backward(pred, target, seq_id)
        return loss.view(())

    @staticmethod
    def backward(ctx, dloss):
        pred, target, seq_id = ctx.saved_tensors
        grad = api.masked_mse_loss_bwd(pred, target, seq_id, dloss.reshape(1).contiguous())
        return grad, None, None


def frame_valid_mse(pred, target, seq_id):
    """Squared-error loss of bf16 pred [B, L, C] against target, averaged
    over the valid tokens (seq_id >= 0: the valid frames), differentiable in
    pred ("lingbot_va_packing" §2.1, compute_loss).  The backward reads pred
    and target again and scales by the incoming gradient on the device."""
    return _MaskedMSE.apply(pred, target, seq_id)

