"""Forward and backward against the fp64 oracle on the whole of workloads 2-5
(GPU).

- Workloads 2 (same-length batch), 3 (padded batch 119/177/285/239 -> 288)
  and 4 (the 64k-token concatenated pack, the size and launch configuration
  bench.py times): every one of the 12 heads, O, LSE, dQ, dK, dV.
- Workload 5 (the length-bucketed sweep): every one of its 40 batches, on
  head i % 12 for batch i.

Each comparison uses the masked-attention parity bar (max |err| <= 2e-2 and
relative L2 <= 1e-2 on valid rows, LSE within 1e-3, padding rows exactly
0 and LSE exactly -inf).  The oracle runs in a pool of worker processes
that start on all jobs as soon as this module's first test asks for the
pool, so the fp64 work overlaps itself and the GPU work.
"""

import numpy as np
import pytest
import torch

import oracle_jobs
import workloads as wl
from attn_check import check_lse, check_rows, to_np

pytestmark = pytest.mark.gpu

HEADS = 12
N_BUCKETS = 40
CONFIGS = (2, 3, 4)


def jobs():
    """Every (layout, heads) the module compares, in the order its tests run."""
    out = [(("config", n), [h]) for n in CONFIGS for h in range(HEADS)]
    out += [(("bucket", i), [i % HEADS]) for i in range(N_BUCKETS)]
    return out


# bound on the wait for one oracle result (the whole pool needs ~2-4 minutes)
RESULT_TIMEOUT_S = 1200


@pytest.fixture(scope="module")
def oracle_results(cuda_ok):
    ex, futures = oracle_jobs.submit_all(jobs())
    try:
        yield futures
    finally:
        for f in futures.values():
            f.cancel()
        ex.shutdown(wait=True, cancel_futures=True)


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def gpu_fwd_bwd(pvl, lay):
    t = wl.make_tensors(lay)
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    tm = pvl.tile_map_build(sid)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = pvl.masked_attn_fwd(q, k, v, sid, tm)
    dq, dk, dv = pvl.masked_attn_bwd(q, k, v, o, do, lse, sid, tm)
    pvl.device_error()
    outs = {"O": o, "LSE": lse, "dQ": dq, "dK": dk, "dV": dv}
    return sid.cpu().numpy(), {name: x.cpu() for name, x in outs.items()}


def compare_head(got: dict, sid: np.ndarray, h: int, result):
    ref_sid, O, LSE, dQ, dK, dV = result
    np.testing.assert_array_equal(sid, ref_sid)
    valid = sid >= 0
    sl = slice(h, h + 1)
    check_rows(f"O[h={h}]", to_np(got["O"][:, :, sl]), O, valid)
    check_lse(to_np(got["LSE"][:, sl]), LSE, valid)
    for name, ref in (("dQ", dQ), ("dK", dK), ("dV", dV)):
        check_rows(f"{name}[h={h}]", to_np(got[name][:, :, sl]), ref, valid)


@pytest.mark.parametrize("n", CONFIGS)
def test_workload_every_head(pvl, oracle_results, n):
    lay = wl.config_layout(n)
    assert lay.H == HEADS
    sid, got = gpu_fwd_bwd(pvl, lay)
    for h in range(HEADS):
        compare_head(got, sid, h, oracle_results[(("config", n), (h,))].result(RESULT_TIMEOUT_S))


@pytest.mark.parametrize("i", range(N_BUCKETS))
def test_bucket_sweep_every_batch(pvl, oracle_results, i):
    lay = wl.bucket_sweep_layouts()[0][i]
    assert lay.H == HEADS
    sid, got = gpu_fwd_bwd(pvl, lay)
    compare_head(got, sid, i % HEADS, oracle_results[(("bucket", i), (i % HEADS,))].result(RESULT_TIMEOUT_S))
