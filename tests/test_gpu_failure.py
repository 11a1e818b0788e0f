"""Failure detection on the GPU without a fault: a bounded wait runs out on
a barrier that nothing arrives on, the kernel records the timeout and
returns, a second warp leaves through the CTA's abort flag, the host reads
PVL_ERR_TIMEOUT with the site, and the context stays usable."""

import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

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
