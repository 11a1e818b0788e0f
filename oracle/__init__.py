"""fp64 CPU oracle for packed variable-length masked attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library and its Python binding) never imports, calls or links it,
and this package imports nothing from the product path; both sides share only
the seeded input generators in ``workloads``.

What it computes, written from the LingBot-VA packing reports:

- ``seq_ids.build_seq_ids``: per-token episode id, -1 for frames at or past
  ``valid_frames`` and for the tail ("lingbot_va_packing" §2.1, FlexAttnFunc
  init_mask; "furniture_packing_variable_length", attention masking).
- ``tile_map.build_tile_map``: empty / partial / full class of every
  (q-tile, k-tile) pair from per-tile seq_id min/max/count, plus compacted
  per-tile lists and the longest-first work order ("lingbot_va_packing" §2.2,
  the block mask built from seq_ids).
- ``attention.attention_fwd`` / ``attention.attention_bwd``: softmax attention
  in which query i attends key j iff seq_id[i] == seq_id[j] >= 0, and its
  analytic gradient ("furniture_packing_variable_length", the seq_id = -1
  masking paragraph; "lingbot_va_attn_profiling", doc_id[q] == doc_id[k]).
- ``loss.masked_mse`` / ``loss.masked_mse_grad``: the squared-error loss
  averaged over valid frames only (frame_valid = f < valid_frames[b]), and
  its gradient ("lingbot_va_packing" §2.1, compute_loss;
  "furniture_packing_variable_length", the loss paragraph).
- ``adaptive_load``: the dual-constraint batch size max(1, min(floor(M_mem/S),
  floor(M_comp/S^p))), the least-squares fit of step_time ~ a + b B S^p by
  brute force over p, the bucket split and the balance measures (coefficient
  of variation, synchronous data-parallel throughput) ("AdaptiveLoad" §2.A, §4).
- ``adaln.adaln_fwd`` / ``adaln.adaln_bwd``: layer norm over the feature
  dimension followed by the AdaLN modulation y = xh (1 + scale) + shift, and
  its gradient with the modulation gradients summed over the sequence
  ("AdaptiveLoad" §2.B, the fused LayerNorm-Modulate kernel).

Every function is pinned by tests under ``tests/`` against brute force,
finite differences, closed forms, library routines (torch fp64 autograd and
scaled_dot_product_attention) and the pages' packed == separate invariant.
"""

from .adaln import adaln_bwd, adaln_fwd  # noqa: F401
from .attention import attention_bwd, attention_fwd, effective_pairs  # noqa: F401
from .loss import frame_valid_tokens, masked_mse, masked_mse_grad, valid_from_seq_id  # noqa: F401
from .seq_ids import build_seq_ids  # noqa: F401
from .tile_map import EMPTY, FULL, PARTIAL, build_tile_map, tile_stats  # noqa: F401
