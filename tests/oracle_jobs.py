"""fp64 oracle jobs for the workload parity tests, run in worker processes.

A job regenerates one workload's seeded inputs from its layout (the
generators in workloads/, which hold none of the method's arithmetic) and
runs the oracle's forward and backward on the listed heads.  Nothing a kernel
produced enters a job.  The workers are started with the spawn method (never
forked from a process that has used CUDA) and run one BLAS thread each, so
that many jobs share the host cores side by side: most of the oracle's time
is elementwise numpy work that one thread does anyway.
"""

from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def layout(spec):
    """("config", n) for workloads 1-4, ("bucket", i) for batch i of workload 5."""
    import workloads as wl
    kind, n = spec
    if kind == "config":
        return wl.config_layout(n)
    if kind == "bucket":
        return wl.bucket_sweep_layouts()[0][n]
    raise ValueError(f"unknown layout {spec!r}")


def fwd_bwd(spec, heads):
    """(seq_id, O, LSE, dQ, dK, dV) of the oracle for layout ``spec`` on ``heads``."""
    import oracle
    import workloads as wl
    lay = layout(spec)
    t = wl.make_tensors(lay)
    sid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    O, LSE = oracle.attention_fwd(t["q"], t["k"], t["v"], sid, heads=heads)
    dQ, dK, dV, _ = oracle.attention_bwd(t["q"], t["k"], t["v"], t["do"], sid, heads=heads)
    return sid, O, LSE, dQ, dK, dV


def submit_all(jobs, workers: int | None = None):
    """Starts a spawn-method pool of single-BLAS-thread workers (one core is
    left to the test process itself) and submits every (spec, heads) job of
    ``jobs`` to fwd_bwd.  Returns (executor, {(spec, tuple(heads)): future}).
    A worker that dies fails its futures (BrokenProcessPool) instead of
    being replaced, so nothing waits forever on a lost job."""
    if workers is None:
        workers = max(1, min(15, (os.cpu_count() or 2) - 1))
    saved = {k: os.environ.get(k) for k in BLAS_ENV}
    os.environ.update({k: "1" for k in BLAS_ENV})
    try:   # the workers start at the first submission and copy this environment
        ex = cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"))
        futures = {(spec, tuple(heads)): ex.submit(fwd_bwd, spec, list(heads)) for spec, heads in jobs}
    finally:   # this process keeps its own
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return ex, futures
