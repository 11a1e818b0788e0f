"""AdaptiveLoad's shape benchmarking on the library's own kernels (GPU): the
cost model step_time ~ a + b B S^p fitted to measured layer steps explains
them, and dual-constraint batches have a more even modelled load and more
even measured step times than equal-token batches of the same episodes
("AdaptiveLoad" §2.A, §4)."""

import math

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def test_fit_and_balance_on_measured_steps(pvl):
    from packed_variable_length_gb300 import adaptive_load as al
    H, D, T, n_max = 12, 128, 38, 65536
    C = H * D
    g = torch.Generator().manual_seed(5)
    buf = {k: torch.randn(n_max * C, generator=g).to(torch.bfloat16).cuda() for k in ("q", "k", "v", "do")}
    out = {k: torch.empty(n_max * C, dtype=torch.bfloat16, device="cuda") for k in ("o", "dq", "dk", "dv", "y", "dx")}
    shift = torch.zeros(16, C, device="cuda")
    scale = torch.zeros(16, C, device="cuda")

    def step_time(frames, f_pad, reps=3):
        B, L = len(frames), T * f_pad
        v = lambda t: t[: B * L * C].view(B, L, H, D)  # noqa: E731
        q, k, vv, do = (v(buf[n]) for n in ("q", "k", "v", "do"))
        o, dq, dk, dv = (v(out[n]) for n in ("o", "dq", "dk", "dv"))
        sid = pvl.pack_build_seq_ids(np.full((B, 1), f_pad), np.asarray(frames).reshape(B, 1), T, L)
        tm = pvl.tile_map_build(sid)
        x = q.view(B, L, C)

        def run():
            o_, lse = pvl.masked_attn_fwd(q, k, vv, sid, tm, o=o)
            pvl.masked_attn_bwd(q, k, vv, o_, do, lse, sid, tm, dq=dq, dk=dk, dv=dv)
            pvl.adaln_fwd(x, shift[:B], scale[:B], 1e-6, y=out["y"][: B * L * C].view(B, L, C))
            pvl.adaln_bwd(x, scale[:B], do.view(B, L, C), 1e-6, dx=out["dx"][: B * L * C].view(B, L, C))
        run()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e-3)
        pvl.device_error()
        return float(np.median(ts))

    shapes = [(Bn, fp) for fp in (104, 200, 296) for Bn in (1, 2, 4, 8) if Bn * T * fp <= n_max]
    Bs, Ss, ts = (np.array(c, dtype=float) for c in zip(*[(Bn, T * fp, step_time([fp] * Bn, fp)) for Bn, fp in shapes]))
    model = al.fit_cost_model(Bs, Ss, ts)
    assert model.r2 > 0.98, model
    assert 1.0 < model.p < 2.5, model
    assert np.abs(model.predict(Bs, Ss) - ts).max() < 0.25 * ts.max()

    lengths = wl.bucket_sweep_lengths(77, 400)
    m_comp = al.m_comp_for(n_max, T * 104, model.p)
    cv, cv_load = {}, {}
    for name, mc in (("equal_token", math.inf), ("dual", m_comp)):
        batches = al.DualConstraintBatchSampler(lengths, T, n_max, mc, model.p, seed=77).all_batches()
        times, loads = [], []
        for bt in batches:
            frames = [int(lengths[i]) for i in bt]
            fp = int(al.padded_frames(max(frames), 8))
            times.append(step_time(frames, fp, reps=1))
            loads.append(len(bt) * (T * fp) ** model.p)
        cv[name] = al.coefficient_of_variation(times)
        cv_load[name] = al.coefficient_of_variation(loads)
    assert cv_load["dual"] < 0.8 * cv_load["equal_token"], cv_load
    assert cv["dual"] < cv["equal_token"], cv
