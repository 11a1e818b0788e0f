"""seq_id and tile-map kernels against the oracle, bit for bit (GPU)."""

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def gpu_seq_ids(pvl, lay):
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    torch.cuda.synchronize()
    return sid


def compare_tile_maps(got: dict, ref: dict):
    for key in ("q_nv", "q_lo", "q_hi", "k_nv", "k_lo", "k_hi", "cls", "row_count", "row_full", "row_list",
                "col_count", "col_full", "col_list", "q_order", "k_order"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    assert list(got["header"][:9]) == [0x544C5650, 2, ref["B"], ref["L"], ref["block_m"], ref["block_n"],
                                       ref["nTq"], ref["nTk"], ref["Lk"]]


def layouts():
    out = [wl.config_layout(n) for n in (1, 2, 3, 4)]
    sweep, _, _ = wl.bucket_sweep_layouts()
    out += sweep          # all 40 batches of workload 5
    rng = np.random.default_rng(77)
    for i in range(6):
        out.append(wl.random_layout(rng, B=3, K=int(rng.integers(1, 6)), T=int(rng.integers(1, 40)),
                                    L=int(rng.integers(1, 3000)), H=1, D=64, name=f"rand{i}"))
    return out


@pytest.mark.parametrize("lay", layouts(), ids=lambda l: l.name)
def test_seq_ids_and_tile_map_bit_exact(pvl, lay):
    sid = gpu_seq_ids(pvl, lay)
    ref_sid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    np.testing.assert_array_equal(sid.cpu().numpy(), ref_sid)
    tm = pvl.tile_map_build(sid, 128, 128)
    torch.cuda.synchronize()
    compare_tile_maps(tm.to_host(0), oracle.build_tile_map(ref_sid, lay.L, 128, 128))
    compare_tile_maps(tm.to_host(1), oracle.build_tile_map(ref_sid, lay.L, 256, 128))


@pytest.mark.parametrize("seed,bm,bn", [(0, 8, 8), (1, 16, 8), (2, 8, 32), (3, 64, 128), (4, 1, 1)])
def test_tile_map_interleaved_ids(pvl, seed, bm, bn):
    rng = np.random.default_rng(seed)
    B, L = 3, int(rng.integers(5, 400))
    ids = rng.integers(-1, 6, size=(B, L)).astype(np.int32)
    sid = torch.from_numpy(ids).cuda()
    tm = pvl.tile_map_build(sid, bm, bn)
    torch.cuda.synchronize()
    compare_tile_maps(tm.to_host(0), oracle.build_tile_map(ids, L, bm, bn))
    compare_tile_maps(tm.to_host(1), oracle.build_tile_map(ids, L, 2 * bm, bn))


def test_tile_map_large_order(pvl):
    """Over a thousand tiles: the order sort runs over many keys."""
    lay = wl.random_layout(np.random.default_rng(9), B=4, K=3, T=40, L=20000, H=1, D=64, name="big")
    sid = gpu_seq_ids(pvl, lay)
    ref_sid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    np.testing.assert_array_equal(sid.cpu().numpy(), ref_sid)
    tm = pvl.tile_map_build(sid, 64, 64)
    torch.cuda.synchronize()
    compare_tile_maps(tm.to_host(), oracle.build_tile_map(ref_sid, lay.L, 64, 64))


def test_seq_ids_rejects_bad_tables(pvl):
    with pytest.raises(pvl.PvlError):
        pvl.pack_build_seq_ids([[5]], [[6]], 2, 100)
    with pytest.raises(pvl.PvlError):
        pvl.pack_build_seq_ids([[60]], [[6]], 2, 100)
