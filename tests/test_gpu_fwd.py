"""masked_attn_fwd against the fp64 oracle (GPU)."""

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from attn_check import check_lse, check_rows, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def run_fwd(pvl, lay, t, sid=None):
    if sid is None:
        sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    tm = pvl.tile_map_build(sid)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o, lse = pvl.masked_attn_fwd(q, k, v, sid, tm)
    pvl.device_error()
    return sid.cpu().numpy(), o, lse


def check_against_oracle(pvl, lay, heads=None, sid_override=None):
    t = wl.make_tensors(lay, with_grad_out=False)
    sid_t = None if sid_override is None else torch.from_numpy(sid_override).cuda()
    sid, o, lse = run_fwd(pvl, lay, t, sid_t)
    heads = list(range(lay.H)) if heads is None else heads
    O_ref, LSE_ref = oracle.attention_fwd(t["q"], t["k"], t["v"], sid, heads=heads)
    valid = sid >= 0
    st = check_rows("O", to_np(o)[:, :, heads], O_ref, valid)
    check_lse(to_np(lse)[:, heads], LSE_ref, valid)
    return st


def test_tiny_workload(pvl):
    """Workload 1, every head (workloads 2-5 in full: test_gpu_workload_parity.py)."""
    check_against_oracle(pvl, wl.config_layout(1))


def random_layouts():
    rng = np.random.default_rng(2024)
    out = []
    for i, (L, D) in enumerate([(1, 64), (100, 128), (129, 64), (300, 128), (777, 64), (1000, 128),
                                (1500, 128), (2049, 64)]):
        lay = wl.random_layout(rng, B=int(rng.integers(1, 4)), K=int(rng.integers(1, 5)),
                               T=int(rng.integers(1, 45)), L=L, H=2, D=D, name=f"rand{i}_L{L}_D{D}")
        out.append(lay)
    return out


@pytest.mark.parametrize("lay", random_layouts(), ids=lambda l: l.name)
def test_random_layouts(pvl, lay):
    check_against_oracle(pvl, lay)


@pytest.mark.parametrize("D", [64, 128])
def test_interleaved_ids(pvl, D):
    """Non-contiguous ids: almost every tile is PARTIAL, the mask does all the work."""
    rng = np.random.default_rng(D)
    B, L = 2, 700
    sid = rng.integers(-1, 4, size=(B, L)).astype(np.int32)
    lay = wl.configs._layout("interleaved", [[0]] * B, [[0]] * B, 1, L, 3, D, 55)
    check_against_oracle(pvl, lay, sid_override=sid)


def test_all_padding_row_and_empty_tiles(pvl):
    lay = wl.configs._layout("pad", [[10], [0], [3]], [[0], [0], [3]], 20, 600, 2, 128, 66)
    check_against_oracle(pvl, lay)


def test_guard_bytes_untouched(pvl):
    lay = wl.random_layout(np.random.default_rng(5), B=2, K=3, T=17, L=900, H=3, D=128)
    t = wl.make_tensors(lay, with_grad_out=False)
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    tm = pvl.tile_map_build(sid)
    n = lay.B * lay.L * lay.H * lay.D
    guard = 4096
    obuf = torch.full((n + guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((lay.B * lay.H * lay.L + guard,), 7.0, dtype=torch.float32, device="cuda")
    o = obuf[:n].view(lay.B, lay.L, lay.H, lay.D)
    lse = lbuf[:lay.B * lay.H * lay.L].view(lay.B, lay.H, lay.L)
    pvl.masked_attn_fwd(t["q"].cuda(), t["k"].cuda(), t["v"].cuda(), sid, tm, o=o, lse=lse)
    pvl.device_error()
    assert torch.isnan(obuf[n:]).all()
    assert (lbuf[lay.B * lay.H * lay.L:] == 7.0).all()
    assert not torch.isnan(o).any()


def test_deterministic(pvl):
    lay = wl.config_layout(3)
    t = wl.make_tensors(lay, with_grad_out=False)
    _, o1, l1 = run_fwd(pvl, lay, t)
    _, o2, l2 = run_fwd(pvl, lay, t)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_tile_map_of_other_shape_is_rejected_on_device(pvl):
    lay = wl.config_layout(1)
    t = wl.make_tensors(lay, with_grad_out=False)
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    tm = pvl.tile_map_build(sid, 64, 64)   # wrong block size for the attention kernels
    o = torch.full_like(t["q"].cuda(), 3.0)
    with pytest.raises(pvl.PvlError) as ei:
        pvl.masked_attn_fwd(t["q"].cuda(), t["k"].cuda(), t["v"].cuda(), sid, tm, o=o)
        pvl.device_error()
    assert ei.value.status == 1
    assert (o == 3.0).all()
    pvl.device_error()   # the record was cleared
