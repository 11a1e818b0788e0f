"""The bench's pipelined end-to-end loop (GPU): with neighbouring steps'
copies overlapping the compute, every step still reads its own inputs and
returns its own results.  Each step gets different inputs (a per-step
scale of the same tensors) and its copied-back outputs must equal those of a
plain synchronous call."""

import numpy as np
import pytest
import torch

import bench
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def test_pipelined_steps_keep_their_own_data(pvl):
    lay = wl.config_layout(2)
    host = wl.make_tensors(lay)
    n_steps = 5
    T, L = lay.tokens_per_frame, lay.L
    # step i's inputs: the drawn tensors scaled by a per-step factor (exact in bf16)
    factors = [1.0, 0.5, 2.0, 0.25, 4.0]
    pinned = [{k: (v.float() * f).to(torch.bfloat16).pin_memory() for k, v in host.items()} for f in factors]
    sets_in = [{k: torch.empty(v.shape, dtype=v.dtype, device="cuda") for k, v in host.items()} for _ in range(2)]
    sets_out = [{"o": torch.empty(host["q"].shape, dtype=torch.bfloat16, device="cuda"),
                 "dq": torch.empty(host["q"].shape, dtype=torch.bfloat16, device="cuda")} for _ in range(2)]
    # one pinned host buffer per step, so no step's results are overwritten
    out_step = [{n: torch.empty(tt.shape, dtype=tt.dtype, pin_memory=True) for n, tt in sets_out[0].items()}
                for _ in range(n_steps)]
    sid = torch.empty((lay.B, L), dtype=torch.int32, device="cuda")
    step_of = {"h2d": 0, "compute": 0, "d2h": 0}

    def h2d(b):
        i = step_of["h2d"]
        step_of["h2d"] += 1
        for k in host:
            sets_in[b][k].copy_(pinned[i][k], non_blocking=True)

    def compute(b):
        step_of["compute"] += 1
        di, do_ = sets_in[b], sets_out[b]
        pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, T, L, out=sid)
        tm = pvl.tile_map_build(sid)
        o, lse = pvl.masked_attn_fwd(di["q"], di["k"], di["v"], sid, tm, o=do_["o"])
        pvl.masked_attn_bwd(di["q"], di["k"], di["v"], o, di["do"], lse, sid, tm, dq=do_["dq"])

    def d2h(b):
        i = step_of["d2h"]
        step_of["d2h"] += 1
        for n, tt in sets_out[b].items():
            out_step[i][n].copy_(tt, non_blocking=True)

    bench.pipelined_e2e(n_steps, h2d, compute, d2h)   # returns after a device synchronize
    pvl.device_error()
    assert step_of == {"h2d": n_steps, "compute": n_steps, "d2h": n_steps}
    for i, f in enumerate(factors):
        tt = {k: v.cuda() for k, v in pinned[i].items()}
        sid2 = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, T, L)
        tm = pvl.tile_map_build(sid2)
        o, lse = pvl.masked_attn_fwd(tt["q"], tt["k"], tt["v"], sid2, tm)
        dq, _, _ = pvl.masked_attn_bwd(tt["q"], tt["k"], tt["v"], o, tt["do"], lse, sid2, tm)
        assert torch.equal(out_step[i]["o"], o.cpu()), f"step {i}: O differs"
        np.testing.assert_allclose(out_step[i]["dq"].float().numpy(), dq.cpu().float().numpy(), rtol=0.02, atol=2e-3)
