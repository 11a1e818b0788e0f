"""masked_attn_bwd_no_alloc: the backward for callers that cannot allocate
device memory (a plug-in whose host framework owns the whole memory pool, or a
loop where an allocation's device synchronisation is not allowed).  It uses
the library's static scratch array instead of a caller workspace.

The call goes straight through the C ABI (ctypes) and its gradients are
compared with those of masked_attn_bwd, the entry point that takes a
workspace, and with the fp64 oracle, within the parity tolerances, on two
calls in a row (the second call finds the first call's contents in the
shared scratch).  The two entry points run the same kernels, so the oracle
comparison is what would catch a fault they share.  This file is
collected last, so a run that stops at the first failure has run every other
test before it (GPU)."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from attn_check import check_rows, to_np

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20  # PVL_NO_ALLOC_SCRATCH_BYTES in include/pvl.h


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def call_no_alloc(lib, q, k, v, o, do, lse, sid, tm, scale, dq, dk, dv):
    B, L, H, D = q.shape
    return lib.masked_attn_bwd_no_alloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                        lse.data_ptr(), sid.data_ptr(), tm.ws.data_ptr(), B, L, H, D,
                                        ctypes.c_float(scale), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("seed,D", [(31, 128), (32, 64)])
def test_matches_workspace_entry_point_twice(pvl, seed, D):
    from packed_variable_length_gb300 import _lib
    lib = _lib.load()
    lay = wl.random_layout(np.random.default_rng(seed), B=2, K=3, T=19, L=1500, H=3, D=D)
    assert pvl.masked_attn_bwd_ws_bytes(lay.B, lay.L, lay.H, lay.D) <= SCRATCH_BYTES
    t = wl.make_tensors(lay)
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    tm = pvl.tile_map_build(sid)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = pvl.masked_attn_fwd(q, k, v, sid, tm)
    ref = pvl.masked_attn_bwd(q, k, v, o, do, lse, sid, tm)
    pvl.device_error()
    s = sid.cpu().numpy()
    valid = s >= 0
    dQ, dK, dV, _ = oracle.attention_bwd(t["q"], t["k"], t["v"], t["do"], s)
    scale = 1.0 / np.sqrt(D)
    for call in range(2):
        outs = [torch.full_like(q, float("nan")) for _ in range(3)]
        st = call_no_alloc(lib, q, k, v, o, do, lse, sid, tm, scale, *outs)
        assert st == 0, lib.pvl_last_error_message().decode()
        pvl.device_error()
        for name, got, want, exact in zip(("dQ", "dK", "dV"), outs, ref, (dQ, dK, dV)):
            check_rows(f"{name} (call {call + 1})", to_np(got), to_np(want), valid)
            check_rows(f"{name} (call {call + 1}, oracle)", to_np(got), exact, valid)


def test_rejects_shapes_beyond_the_scratch(pvl):
    from packed_variable_length_gb300 import _lib
    lib = _lib.load()
    B, L, H, D = 1, 65536, 12, 128   # needs about 400 MB of scratch
    assert pvl.masked_attn_bwd_ws_bytes(B, L, H, D) > SCRATCH_BYTES
    dummy = 1 << 20                  # never dereferenced: the call returns before launching
    st = lib.masked_attn_bwd_no_alloc(dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, B, L, H, D,
                                      ctypes.c_float(0.088), dummy, dummy, dummy, None)
    assert st == 2
    assert b"static scratch" in lib.pvl_last_error_message()
