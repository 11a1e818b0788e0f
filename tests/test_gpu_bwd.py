"""masked_attn_bwd against the fp64 oracle (GPU).  The kernels' forward
produces O and LSE; the oracle recomputes everything from Q, K, V, dO."""

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from attn_check import check_rows, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def run_fwd_bwd(pvl, lay, t, sid=None, ws_fill=None):
    if sid is None:
        sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    tm = pvl.tile_map_build(sid)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = pvl.masked_attn_fwd(q, k, v, sid, tm)
    ws = None
    if ws_fill is not None:
        nbytes = pvl.masked_attn_bwd_ws_bytes(*q.shape)
        ws = torch.full((nbytes // 4,), ws_fill, dtype=torch.float32, device="cuda").view(torch.uint8)
    dq, dk, dv = pvl.masked_attn_bwd(q, k, v, o, do, lse, sid, tm, ws=ws)
    pvl.device_error()
    return sid.cpu().numpy(), dq, dk, dv


def check_against_oracle(pvl, lay, heads=None, sid_override=None, ws_fill=None):
    t = wl.make_tensors(lay)
    sid_t = None if sid_override is None else torch.from_numpy(sid_override).cuda()
    sid, dq, dk, dv = run_fwd_bwd(pvl, lay, t, sid_t, ws_fill)
    heads = list(range(lay.H)) if heads is None else heads
    dQ, dK, dV, _ = oracle.attention_bwd(t["q"], t["k"], t["v"], t["do"], sid, heads=heads)
    valid = sid >= 0
    out = {}
    for name, got, ref in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
        out[name] = check_rows(name, to_np(got)[:, :, heads], ref, valid)
    return out


def test_tiny_workload(pvl):
    """Workload 1, every head (workloads 2-5 in full: test_gpu_workload_parity.py)."""
    check_against_oracle(pvl, wl.config_layout(1))


def random_layouts():
    rng = np.random.default_rng(4048)
    out = []
    for i, (L, D) in enumerate([(1, 64), (100, 128), (129, 64), (300, 128), (777, 64), (1000, 128),
                                (2049, 128)]):
        out.append(wl.random_layout(rng, B=int(rng.integers(1, 4)), K=int(rng.integers(1, 5)),
                                    T=int(rng.integers(1, 45)), L=L, H=2, D=D, name=f"rand{i}_L{L}_D{D}"))
    return out


@pytest.mark.parametrize("lay", random_layouts(), ids=lambda l: l.name)
def test_random_layouts(pvl, lay):
    check_against_oracle(pvl, lay)


@pytest.mark.parametrize("D", [64, 128])
def test_interleaved_ids(pvl, D):
    rng = np.random.default_rng(D + 1)
    B, L = 2, 700
    sid = rng.integers(-1, 4, size=(B, L)).astype(np.int32)
    lay = wl.configs._layout("interleaved", [[0]] * B, [[0]] * B, 1, L, 3, D, 56)
    check_against_oracle(pvl, lay, sid_override=sid)


def test_all_padding_row_and_empty_tiles(pvl):
    lay = wl.configs._layout("pad", [[10], [0], [3]], [[0], [0], [3]], 20, 600, 2, 128, 67)
    check_against_oracle(pvl, lay)


def test_workspace_contents_are_ignored(pvl):
    lay = wl.random_layout(np.random.default_rng(8), B=2, K=2, T=13, L=700, H=2, D=128)
    check_against_oracle(pvl, lay, ws_fill=float("nan"))


def test_guard_bytes_untouched(pvl):
    lay = wl.random_layout(np.random.default_rng(9), B=2, K=3, T=17, L=900, H=2, D=64)
    t = wl.make_tensors(lay)
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    tm = pvl.tile_map_build(sid)
    q, k, v, do = (t[nm].cuda() for nm in ("q", "k", "v", "do"))
    o, lse = pvl.masked_attn_fwd(q, k, v, sid, tm)
    n = q.numel()
    guard = 4096
    bufs = [torch.full((n + guard,), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    views = [b[:n].view(q.shape) for b in bufs]
    pvl.masked_attn_bwd(q, k, v, o, do, lse, sid, tm, dq=views[0], dk=views[1], dv=views[2])
    pvl.device_error()
    for b, vw in zip(bufs, views):
        assert torch.isnan(b[n:]).all()
        assert not torch.isnan(vw).any()


def test_autograd_wrapper_matches(pvl):
    lay = wl.random_layout(np.random.default_rng(10), B=2, K=2, T=11, L=500, H=2, D=128)
    t = wl.make_tensors(lay)
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    q, k, v = (t[nm].cuda().requires_grad_(True) for nm in ("q", "k", "v"))
    o = pvl.packed_attention(q, k, v, sid)
    o.backward(t["do"].cuda())
    s = sid.cpu().numpy()
    dQ, dK, dV, _ = oracle.attention_bwd(t["q"], t["k"], t["v"], t["do"], s)
    valid = s >= 0
    for name, got, ref in (("dQ", q.grad, dQ), ("dK", k.grad, dK), ("dV", v.grad, dV)):
        check_rows(name, to_np(got), ref, valid)
