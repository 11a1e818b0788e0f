"""Packed variable-length masked attention for GB300 (sm_103a).

Forward and backward self-attention over episodes that are zero-padded to a
shared frame count or concatenated along the sequence axis; a query attends a
key iff both carry the same non-negative seq_id.  The compute runs in
hand-written CUDA kernels (tcgen05 / TMEM / TMA) inside libpvl.so, behind the
C ABI declared in include/pvl.h; this package only marshals arguments.
"""

from .api import (  # noqa: F401
    EMPTY,
    FULL,
    PARTIAL,
    PvlError,
    TileMap,
    adaln_bwd,
    adaln_bwd_ws_bytes,
    adaln_fwd,
    device_error,
    masked_attn_bwd,
    masked_attn_bwd_no_alloc,
    masked_attn_bwd_ws_bytes,
    masked_attn_fwd,
    masked_mse_loss,
    masked_mse_loss_bwd,
    masked_mse_ws_bytes,
    mark_next_bwd_main,
    pack_build_seq_ids,
    set_attn_wait_timeout_ns,
    tile_map_build,
    tile_map_ws_bytes,
    version,
)
from . import adaptive_load  # noqa: F401  (host-side dual-constraint bucketing)
from .autograd import adaln_modulate, frame_valid_mse, packed_attention  # noqa: F401
