"""ctypes loader for libpvl.so: argument and return types of every C entry point.

The library is built in-tree (packed_variable_length_gb300/libpvl.so).  There
is no fallback: if the library is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpvl.so")

_c_int = ctypes.c_int
_c_size = ctypes.c_size_t
_c_float = ctypes.c_float
_p = ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/pvl.h
SIGNATURES = {
    "pack_build_seq_ids": (_c_int, [_p, _p, _c_int, _c_int, _c_int, _c_int, _p, _p]),
    "tile_map_ws_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "tile_map_layout": (_c_int, [_c_int, _c_int, _c_int, _c_int, _p]),
    "tile_map_build": (_c_int, [_p, _c_int, _c_int, _c_int, _c_int, _p, _c_size, _p]),
    "masked_attn_fwd": (_c_int, [_p, _p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int, _c_float, _p, _p, _p]),
    "masked_attn_bwd_ws_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "masked_attn_bwd": (_c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int, _c_float,
                                 _p, _p, _p, _p, _c_size, _p]),
    "masked_attn_bwd_no_alloc": (_c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int,
                                          _c_float, _p, _p, _p, _p]),
    "tile_map_ws_bytes_cross": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "tile_map_layout_cross": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _p]),
    "tile_map_build_cross": (_c_int, [_p, _p, _c_int, _c_int, _c_int, _c_int, _c_int, _p, _c_size, _p]),
    "masked_attn_fwd_cross": (_c_int, [_p, _p, _p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                       _p, _p, _p]),
    "masked_attn_bwd_ws_bytes_cross": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "masked_attn_bwd_cross": (_c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int, _c_int,
                                       _c_float, _p, _p, _p, _p, _c_size, _p]),
    "adaln_fwd": (_c_int, [_p, _p, _p, _c_int, _c_int, _c_int, _c_float, _p, _p, _p, _p]),
    "adaln_bwd_ws_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "adaln_bwd": (_c_int, [_p, _p, _p, _c_int, _c_int, _c_int, _c_float, _p, _p, _p, _p, _c_size, _p]),
    "masked_mse_ws_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "masked_mse_loss": (_c_int, [_p, _p, _p, _c_int, _c_int, _c_int, _p, _p, _c_float, _p, _c_size, _p]),
    "masked_mse_loss_bwd": (_c_int, [_p, _p, _p, _c_int, _c_int, _c_int, _p, _p, _p, _c_size, _p]),
    "pvl_selftest_wait_timeout": (_c_int, [ctypes.c_uint64, ctypes.c_uint64, _p, _p]),
    "pvl_set_attn_wait_timeout_ns": (_c_int, [ctypes.c_uint64]),
    "pvl_mark_next_bwd_main": (_c_int, [_p, _p]),
    "pvl_device_error": (_c_int, [_p]),
    "pvl_device_error_detail": (_c_int, [_p, _p]),
    "pvl_last_error_message": (ctypes.c_char_p, []),
    "pvl_version": (_c_int, []),
}

_lib = None


def load() -> ctypes.CDLL:
    """Loads libpvl.so once; raises RuntimeError when it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m packed_variable_length_gb300.build` "
                "(or __graft_entry__.build()); there is no non-CUDA fallback")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
