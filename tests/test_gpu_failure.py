"""Failure detection on the GPU without a fault.

1. The self-test kernel: a bounded wait runs out on a barrier that nothing
   arrives on, the kernel records the timeout and returns, a second warp
   leaves through the CTA's abort flag, the host reads PVL_ERR_TIMEOUT with
   the site, and the context stays usable.
2. The attention kernels themselves: with the wait bound set to a few
   nanoseconds, far below the microseconds a tile load or a tile's MMAs
   take, their waits on real copies and MMAs run out.  The padded workload
   (B = 4, L = 10944, 12 heads) gives every CTA many such waits; on the tiny
   workload a wait can finish within the device timer's resolution and never
   run out.  Each kernel then takes its abort path (the producer drains its
   copies in flight, the MMA threads wait for their MMAs, tensor memory is
   released), the host reads PVL_ERR_TIMEOUT with a site of that kernel, and
   the same context, with the default bound back, computes the tiny workload
   to the oracle's tolerances and repeats the padded workload's forward bit
   for bit."""

import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from attn_check import check_lse, check_rows, to_np

pytestmark = pytest.mark.gpu

PVL_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def test_bounded_wait_times_out_and_the_context_survives(pvl):
    from packed_variable_length_gb300 import _lib
    lib = _lib.load()
    pvl.device_error()                                  # start from a clear record
    out = (ctypes.c_int32 * 2)(-1, -1)
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    st = lib.pvl_selftest_wait_timeout(50_000_000, 5_000_000_000, ctypes.addressof(out), stream)
    dt = time.perf_counter() - t0
    assert st == 0
    assert list(out) == [0, 0]                          # both waits gave up
    assert dt < 2.0                                     # warp 1 left through the abort flag, not its 5 s limit
    st, info = pvl.device_error(raise_on_error=False)
    assert st == PVL_ERR_TIMEOUT
    assert info[0] == 1 and info[1] == 91               # timeout code, site of the short wait
    assert pvl.device_error(raise_on_error=False)[0] == 0   # reading cleared it
    # the context still runs the path and gets the right answer
    lay = wl.config_layout(1)
    t = wl.make_tensors(lay)
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    tm = pvl.tile_map_build(sid)
    o, lse = pvl.masked_attn_fwd(t["q"].cuda(), t["k"].cuda(), t["v"].cuda(), sid, tm)
    pvl.device_error()
    O, _ = oracle.attention_fwd(t["q"], t["k"], t["v"], sid.cpu().numpy())
    valid = sid.cpu().numpy() >= 0
    err = np.abs(o.double().cpu().numpy()[valid] - O[valid]).max()
    assert err < 2e-2


FWD_SITES = range(1, 15)    # the forward kernel's wait sites
BWD_SITES = range(21, 37)   # the main backward kernel's wait sites


@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_attention_kernel_wait_runs_out_and_the_context_survives(pvl, which):
    big = wl.config_layout(3)
    tb = wl.make_tensors(big)
    sid_b = pvl.pack_build_seq_ids(big.seg_frames, big.seg_valid, big.tokens_per_frame, big.L)
    tm_b = pvl.tile_map_build(sid_b)
    qb, kb, vb, dob = (tb[n].cuda() for n in ("q", "k", "v", "do"))
    pvl.device_error()
    ob, lseb = pvl.masked_attn_fwd(qb, kb, vb, sid_b, tm_b)    # default bound
    pvl.device_error()
    t0 = time.perf_counter()
    try:
        pvl.set_attn_wait_timeout_ns(2)
        if which == "fwd":
            pvl.masked_attn_fwd(qb, kb, vb, sid_b, tm_b, o=torch.empty_like(qb))
        else:
            pvl.masked_attn_bwd(qb, kb, vb, ob, dob, lseb, sid_b, tm_b)
        st, info = pvl.device_error(raise_on_error=False)
    finally:
        pvl.set_attn_wait_timeout_ns(0)
    dt = time.perf_counter() - t0
    assert st == PVL_ERR_TIMEOUT
    assert info[0] == 1 and info[1] in (FWD_SITES if which == "fwd" else BWD_SITES), info
    assert dt < 10.0                                    # every wait on the way out is bounded
    assert pvl.device_error(raise_on_error=False)[0] == 0
    # the same context, default bound: the padded forward again, bit for bit
    ob2, lseb2 = pvl.masked_attn_fwd(qb, kb, vb, sid_b, tm_b)
    pvl.device_error()
    assert torch.equal(ob, ob2) and torch.equal(lseb, lseb2)
    # and the whole path on the tiny workload against the oracle
    lay = wl.config_layout(1)
    t = wl.make_tensors(lay)
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    tm = pvl.tile_map_build(sid)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    s = sid.cpu().numpy()
    valid = s >= 0
    o2, lse2 = pvl.masked_attn_fwd(q, k, v, sid, tm)
    dq, dk, dv = pvl.masked_attn_bwd(q, k, v, o2, do, lse2, sid, tm)
    pvl.device_error()
    O, LSE = oracle.attention_fwd(t["q"], t["k"], t["v"], s)
    dQ, dK, dV, _ = oracle.attention_bwd(t["q"], t["k"], t["v"], t["do"], s)
    check_rows("O", to_np(o2), O, valid)
    check_lse(to_np(lse2), LSE, valid)
    for name, got, ref in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
        check_rows(name, to_np(got), ref, valid)
