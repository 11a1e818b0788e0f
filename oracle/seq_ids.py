"""Oracle: per-token seq_id from a segment table.  TEST INFRASTRUCTURE ONLY.

"lingbot_va_packing" §2.1 (wan_va/modules/model.py, FlexAttnFunc.init_mask
with valid_frames): the latent/action seq_id of a token whose frame index is
>= valid_frames[b] becomes -1, which removes it from the attention mask.
"furniture_packing_variable_length" (masking paragraph) repeats this: padding
tokens get seq_id -1 and so drop out on both the query and the key side.
"lingbot_va_attn_profiling" (packing proposal) tags concatenated episodes with
a per-token document id.

Segment table reading used here: row b holds K segments laid end to end; the
segment k covers seg_frames[b, k] frames of tokens_per_frame tokens each; its
first seg_valid[b, k] frames are real and carry id b * K + k; its remaining
frames and every position after the last segment (up to L) carry -1.
"""

from __future__ import annotations

import numpy as np


def build_seq_ids(seg_frames, seg_valid, tokens_per_frame: int, L: int) -> np.ndarray:
    seg_frames = np.asarray(seg_frames, dtype=np.int64)
    seg_valid = np.asarray(seg_valid, dtype=np.int64)
    if seg_frames.ndim != 2 or seg_frames.shape != seg_valid.shape:
        raise ValueError("seg_frames and seg_valid must both be [B, K]")
    if tokens_per_frame <= 0 or L <= 0:
        raise ValueError("tokens_per_frame and L must be positive")
    if (seg_frames < 0).any() or (seg_valid < 0).any() or (seg_valid > seg_frames).any():
        raise ValueError("need 0 <= seg_valid <= seg_frames")
    B, K = seg_frames.shape
    out = np.full((B, L), -1, dtype=np.int32)
    for b in range(B):
        if int(seg_frames[b].sum()) * tokens_per_frame > L:
            raise ValueError(f"row {b}: segments need more than L={L} tokens")
        pos = 0
        for k in range(K):
            for f in range(int(seg_frames[b, k])):
                if f < seg_valid[b, k]:
                    out[b, pos:pos + tokens_per_frame] = b * K + k
                pos += tokens_per_frame
    return out
