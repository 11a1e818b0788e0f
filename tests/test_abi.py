"""The C ABI without a GPU: libpvl.so loads and exports every symbol that
include/pvl.h declares; host-side validation rejects bad arguments before any
device work (CPU only)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "pvl.h")).read()
    return re.findall(r"PVL_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


@pytest.fixture(scope="module")
def lib():
    from packed_variable_length_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        try:
            build.build()
        except RuntimeError as e:  # no toolkit on this machine
            pytest.skip(str(e))
    return _lib.load()


def test_header_declares_the_four_calls():
    syms = declared_symbols()
    for name in ("pack_build_seq_ids", "tile_map_build", "masked_attn_fwd", "masked_attn_bwd"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    from packed_variable_length_gb300 import _lib
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"
    assert set(_lib.SIGNATURES) == set(declared_symbols())


def test_only_declared_symbols_are_exported(lib):
    from packed_variable_length_gb300 import _lib
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    names = {ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln}
    ours = {n for n in names if n.startswith(("pvl_", "pack_", "tile_map", "masked_attn", "masked_mse", "adaln_"))}
    assert ours == set(declared_symbols())


def test_host_validation_without_gpu(lib):
    null = None
    assert lib.pack_build_seq_ids(null, null, 1, 1, 1, 1, null, null) == 1
    frames = (ctypes.c_int32 * 1)(5)
    valid = (ctypes.c_int32 * 1)(6)      # valid > frames
    dummy = ctypes.c_void_p(256)
    assert lib.pack_build_seq_ids(ctypes.addressof(frames), ctypes.addressof(valid), 1, 1, 2, 100, dummy, null) == 1
    valid[0] = 5
    assert lib.pack_build_seq_ids(ctypes.addressof(frames), ctypes.addressof(valid), 1, 1, 40, 100, dummy, null) == 1
    assert b"tokens" in lib.pvl_last_error_message()
    # D outside {64, 128}
    assert lib.masked_attn_fwd(dummy, dummy, dummy, dummy, dummy, 1, 128, 1, 96, 0.1, dummy, dummy, null) == 2
    assert lib.masked_attn_bwd(dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, 1, 128, 1, 64, 0.1,
                               dummy, dummy, dummy, dummy, 0, null) == 1   # short workspace
    assert lib.tile_map_build(null, 1, 1, 128, 128, null, 0, null) == 1
    assert lib.tile_map_ws_bytes(0, 10, 128, 128) == 0
    # cross attention: key length checked on its own side
    assert lib.masked_attn_fwd_cross(dummy, dummy, dummy, dummy, dummy, dummy, 1, 128, 0, 1, 64, 0.1, dummy,
                                     dummy, null) == 1
    assert lib.tile_map_build_cross(dummy, null, 1, 10, 10, 128, 128, dummy, 1 << 20, null) == 1
    assert lib.tile_map_ws_bytes_cross(1, 10, 0, 128, 128) == 0
    assert lib.tile_map_ws_bytes_cross(2, 1000, 300, 128, 128) < lib.tile_map_ws_bytes(2, 1000, 128, 128)
    # AdaLN: D must be a multiple of 8 up to 8192; eps >= 0; workspace size
    assert lib.adaln_fwd(dummy, dummy, dummy, 1, 4, 100, 1e-6, dummy, null, null, null) == 2
    assert lib.adaln_fwd(dummy, dummy, dummy, 1, 4, 8200, 1e-6, dummy, null, null, null) == 2
    assert lib.adaln_fwd(dummy, dummy, dummy, 1, 4, 64, -1.0, dummy, null, null, null) == 1
    assert lib.adaln_bwd(dummy, dummy, dummy, 1, 4, 64, 1e-6, dummy, dummy, dummy, dummy, 0, null) == 1
    assert lib.adaln_bwd_ws_bytes(2, 100, 64) == 2 * (200 + 1) * 64 * 4      # a slot per (CTA, batch row)
    assert lib.adaln_bwd_ws_bytes(1, 64000, 5120) == 2 * 2048 * 5120 * 4     # at most 2048 CTAs
    # bounded-wait self-test: argument checks only (no GPU here)
    out2 = (ctypes.c_int32 * 2)()
    assert lib.pvl_selftest_wait_timeout(0, 10, ctypes.addressof(out2), null) == 1
    assert lib.pvl_selftest_wait_timeout(10, 5, ctypes.addressof(out2), null) == 1
    assert lib.pvl_selftest_wait_timeout(10, 20, null, null) == 1
    # attention wait bound: at most 60 s, 0 restores the default; event marks need no GPU to be set or cleared
    assert lib.pvl_set_attn_wait_timeout_ns(61_000_000_000) == 1
    assert lib.pvl_set_attn_wait_timeout_ns(0) == 0
    assert lib.pvl_mark_next_bwd_main(null, null) == 0
    # masked loss: C a multiple of 8, a finite grad_scale, a full workspace
    ws = lib.masked_mse_ws_bytes(1, 10, 8)
    assert ws > 0 and lib.masked_mse_ws_bytes(0, 10, 8) == 0
    assert lib.masked_mse_loss(dummy, dummy, dummy, 1, 10, 12, dummy, null, 1.0, dummy, ws, null) == 2
    assert lib.masked_mse_loss(null, dummy, dummy, 1, 10, 8, dummy, null, 1.0, dummy, ws, null) == 1
    assert lib.masked_mse_loss(dummy, dummy, dummy, 1, 10, 8, null, null, 1.0, dummy, ws, null) == 1
    assert lib.masked_mse_loss(dummy, dummy, dummy, 1, 10, 8, dummy, null, float("nan"), dummy, ws, null) == 1
    assert lib.masked_mse_loss(dummy, dummy, dummy, 1, 10, 8, dummy, null, 1.0, dummy, ws - 1, null) == 1
    assert lib.masked_mse_loss_bwd(dummy, dummy, dummy, 1, 10, 8, null, dummy, dummy, ws, null) == 1
    assert lib.masked_mse_loss_bwd(dummy, dummy, dummy, 0, 10, 8, dummy, dummy, dummy, ws, null) == 1


def test_tile_map_layout_host(lib):
    import numpy as np
    offs = (ctypes.c_size_t * 32)()
    assert lib.tile_map_layout(2, 1000, 128, 64, ctypes.addressof(offs)) == 0
    o = list(offs)
    assert o[0] == 0 and all(b > a for a, b in zip(o, o[1:])) and all(x % 256 == 0 for x in o)
    total = lib.tile_map_ws_bytes(2, 1000, 128, 64)
    nq, nk = 2 * 8, 2 * 16          # level 0: 128-row query tiles, 64-key tiles
    assert o[8] - o[7] >= nq * 16   # level-0 cls bytes
    assert o[16 + 8] - o[16 + 7] >= 2 * 4 * 16   # level-1 cls: 256-row query tiles
    assert total >= o[-1] + 4 * nk
    assert lib.masked_attn_bwd_ws_bytes(2, 1000, 3, 128) >= 2 * 1000 * 3 * 128 * 4
    assert np.int64(lib.pvl_version()) > 0
