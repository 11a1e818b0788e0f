"""Cross attention (queries and keys with their own seq_ids and lengths,
"lingbot_va_packing" §2.1) against the fp64 oracle (GPU): the rectangular
tile map bit for bit, forward and backward within the parity tolerances."""

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from attn_check import check_lse, check_rows, to_np
from test_gpu_seq_tile import compare_tile_maps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def cross_ids(pvl, cl):
    q = cl.q
    qsid = pvl.pack_build_seq_ids(q.seg_frames, q.seg_valid, q.tokens_per_frame, cl.Lq)
    ksid = pvl.pack_build_seq_ids(q.seg_frames, q.seg_valid, cl.tokens_per_frame_k, cl.Lk)
    return qsid, ksid


def random_cross_layouts():
    rng = np.random.default_rng(5150)
    out = []
    for i, (L, D, Tk, Lk) in enumerate([(300, 128, 3, None), (777, 64, 7, None), (129, 128, 1, 1),
                                        (2049, 128, 11, None), (1000, 64, 20, 4000), (256, 128, 2, 100)]):
        lay = wl.random_layout(rng, B=int(rng.integers(1, 4)), K=int(rng.integers(1, 5)),
                               T=int(rng.integers(1, 40)), L=L, H=2, D=D, name=f"rand{i}_L{L}_D{D}")
        out.append(wl.cross_layout(lay, Tk, Lk))
    return out


def tile_map_layouts():
    return [wl.cross_config_layout(n) for n in (2, 3, 4)] + random_cross_layouts()


@pytest.mark.parametrize("cl", tile_map_layouts(), ids=lambda c: f"{c.name}_Lk{c.Lk}")
def test_cross_tile_map(pvl, cl):
    qsid, ksid = cross_ids(pvl, cl)
    tm = pvl.tile_map_build(qsid, k_seq_id=ksid)
    torch.cuda.synchronize()
    qs, ks = qsid.cpu().numpy(), ksid.cpu().numpy()
    compare_tile_maps(tm.to_host(0), oracle.build_tile_map(qs, cl.Lq, 128, 128, k_seq_id=ks, Lk=cl.Lk))
    compare_tile_maps(tm.to_host(1), oracle.build_tile_map(qs, cl.Lq, 256, 128, k_seq_id=ks, Lk=cl.Lk))


def check_cross(pvl, cl, heads=None, qsid=None, ksid=None):
    t = wl.make_cross_tensors(cl)
    if qsid is None:
        qsid, ksid = cross_ids(pvl, cl)
    else:
        qsid, ksid = torch.from_numpy(qsid).cuda(), torch.from_numpy(ksid).cuda()
    tm = pvl.tile_map_build(qsid, k_seq_id=ksid)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = pvl.masked_attn_fwd(q, k, v, qsid, tm, k_seq_id=ksid)
    dq, dk, dv = pvl.masked_attn_bwd(q, k, v, o, do, lse, qsid, tm, k_seq_id=ksid)
    pvl.device_error()
    assert dk.shape == k.shape and dq.shape == q.shape
    qs, ks = qsid.cpu().numpy(), ksid.cpu().numpy()
    heads = list(range(cl.H)) if heads is None else heads
    O, LSE = oracle.attention_fwd(t["q"], t["k"], t["v"], qs, heads=heads, k_seq_id=ks)
    dQ, dK, dV, _ = oracle.attention_bwd(t["q"], t["k"], t["v"], t["do"], qs, heads=heads, k_seq_id=ks)
    # a query without an admissible key is a padding row; likewise a key no query reaches
    q_ok = np.stack([(qs[b] >= 0) & np.isin(qs[b], ks[b]) for b in range(cl.B)])
    k_ok = np.stack([(ks[b] >= 0) & np.isin(ks[b], qs[b][qs[b] >= 0]) for b in range(cl.B)])
    stats = {"O": check_rows("O", to_np(o)[:, :, heads], O, q_ok)}
    stats["LSE"] = check_lse(to_np(lse)[:, heads], LSE, q_ok)
    stats["dQ"] = check_rows("dQ", to_np(dq)[:, :, heads], dQ, q_ok)
    stats["dK"] = check_rows("dK", to_np(dk)[:, :, heads], dK, k_ok)
    stats["dV"] = check_rows("dV", to_np(dv)[:, :, heads], dV, k_ok)
    return stats


@pytest.mark.parametrize("n,heads", [(2, [0, 7]), (3, [1, 10]), (4, [3])])
def test_cross_workloads(pvl, n, heads):
    check_cross(pvl, wl.cross_config_layout(n), heads)


@pytest.mark.parametrize("cl", random_cross_layouts(), ids=lambda c: f"{c.name}_Lk{c.Lk}")
def test_cross_random_layouts(pvl, cl):
    check_cross(pvl, cl)


@pytest.mark.parametrize("D", [64, 128])
def test_cross_interleaved_ids(pvl, D):
    """Ids drawn per position on both sides; id 4 has queries only, id 5 keys
    only, so some valid queries and keys take no part."""
    rng = np.random.default_rng(D + 3)
    B, Lq, Lk = 2, 700, 333
    lay = wl.configs._layout("interleaved", [[0]] * B, [[0]] * B, 1, Lq, 3, D, 91)
    cl = wl.cross_layout(lay, 1, Lk)
    qsid = rng.integers(-1, 5, size=(B, Lq)).astype(np.int32)
    ksid = rng.integers(-1, 4, size=(B, Lk)).astype(np.int32)
    ksid[ksid == 3] = 5
    check_cross(pvl, cl, qsid=qsid, ksid=ksid)


def test_cross_no_key_is_padding(pvl):
    """Every key id -1: O = 0, LSE = -inf, all gradients 0."""
    lay = wl.configs._layout("nokeys", [[4]], [[4]], 40, 300, 2, 128, 5)
    cl = wl.cross_layout(lay, 8, 200)
    qsid = np.zeros((1, 300), np.int32)
    qsid[0, 160:] = -1
    ksid = np.full((1, 200), -1, np.int32)
    check_cross(pvl, cl, qsid=qsid, ksid=ksid)


def test_cross_with_own_ids_matches_self(pvl):
    """k_seq_id = seq_id, Lk = L through the cross entry points gives the
    self-attention results exactly."""
    lay = wl.config_layout(3)
    t = wl.make_tensors(lay)
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    tm_s = pvl.tile_map_build(sid)
    tm_c = pvl.tile_map_build(sid, k_seq_id=sid.clone())
    o1, l1 = pvl.masked_attn_fwd(q, k, v, sid, tm_s)
    o2, l2 = pvl.masked_attn_fwd(q, k, v, sid, tm_c, k_seq_id=sid.clone())
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = pvl.masked_attn_bwd(q, k, v, o1, do, l1, sid, tm_s)
    g2 = pvl.masked_attn_bwd(q, k, v, o2, do, l2, sid, tm_c, k_seq_id=sid.clone())
    pvl.device_error()
    for a, b in zip(g1[1:], g2[1:]):
        assert torch.equal(a, b)  # dK, dV have no atomics
    for a, b in zip(g1[:1], g2[:1]):
        assert torch.allclose(a.float(), b.float(), atol=2e-3, rtol=0)  # dQ: reduction order varies


def test_cross_autograd(pvl):
    lay = wl.random_layout(np.random.default_rng(9), B=2, K=3, T=5, L=400, H=2, D=64)
    cl = wl.cross_layout(lay, 3)
    t = wl.make_cross_tensors(cl)
    qsid, ksid = cross_ids(pvl, cl)
    q, k, v = (t[n].cuda().requires_grad_() for n in ("q", "k", "v"))
    o = pvl.packed_attention(q, k, v, qsid, k_seq_id=ksid)
    o.backward(t["do"].cuda())
    pvl.device_error()
    dQ, dK, dV, _ = oracle.attention_bwd(t["q"], t["k"], t["v"], t["do"], qsid.cpu().numpy(),
                                         k_seq_id=ksid.cpu().numpy())
    qs, ks = qsid.cpu().numpy(), ksid.cpu().numpy()
    q_ok = np.stack([(qs[b] >= 0) & np.isin(qs[b], ks[b]) for b in range(cl.B)])
    k_ok = np.stack([(ks[b] >= 0) & np.isin(ks[b], qs[b][qs[b] >= 0]) for b in range(cl.B)])
    check_rows("dQ", to_np(q.grad), dQ, q_ok)
    check_rows("dK", to_np(k.grad), dK, k_ok)
    check_rows("dV", to_np(v.grad), dV, k_ok)
