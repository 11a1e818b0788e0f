"""Seeded synthetic inputs for packed variable-length attention.

This package only *draws* inputs: episode lengths, batch composition, segment
layouts (frames and valid frames per segment) and the bf16 tensors Q, K, V and
the upstream gradient dO.  It holds none of the attention arithmetic (no
seq_id construction, no tile classification, no softmax), so both the CUDA path
and the fp64 oracle can consume the same inputs without sharing method code.

The shapes follow the LingBot-VA packing reports ("lingbot_va_packing", §2.1
and §3.1; "furniture_packing_variable_length"): latent frame counts F from 103
to 362, padded to a multiple of 8 latent frames, 38 tokens per latent frame,
up to 64k tokens per packed sequence.  The real FurnitureBench episodes are
replaced by uniform draws of F.
"""

from .configs import (  # noqa: F401
    ACTION_TOKENS_PER_FRAME,
    CrossLayout,
    F_MAX,
    F_MIN,
    PAD_MULTIPLE,
    TOKENS_PER_FRAME,
    Layout,
    bucket_sweep_layouts,
    bucket_sweep_lengths,
    config_layout,
    cross_config_layout,
    cross_layout,
    make_cross_tensors,
    make_loss_tensors,
    make_tensors,
    random_layout,
    round_up,
)
from .sampler import LengthBucketBatchSampler, padding_waste  # noqa: F401
