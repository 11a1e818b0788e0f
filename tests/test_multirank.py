"""The bench's multi-rank path (replicas only: no collective on the data
path) with world_size 2 on gloo, on the CPU: the barrier, the max over ranks
of the step time, the whole-job aggregate, and a rank that fails is seen by
the others through the process group instead of a hang."""

import os
import socket

import pytest


def _port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank(rank, world, port, q, fail_rank):
    import datetime

    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    try:
        bench.barrier(world)
        ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, world)
        value = bench.aggregate(1.0e6, slowest, world)
        if rank == fail_rank:
            raise SystemExit(3)                      # leaves between steps, nothing in flight
        try:
            bench.barrier(world)
            q.put((rank, slowest, value, "ok"))
        except Exception as exc:                     # the others learn of it from the group
            q.put((rank, slowest, value, type(exc).__name__))
    finally:
        try:
            dist.destroy_process_group()
        except Exception:
            pass


def _run(world, fail_rank=-1):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q, fail_rank)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    out = []
    while not q.empty():
        out.append(q.get())
    return sorted(out), [p.exitcode for p in procs]


def test_two_replicas_report_the_slowest_rank():
    out, codes = _run(2)
    assert codes == [0, 0]
    assert [o[0] for o in out] == [0, 1]
    for _, slowest, value, status in out:
        assert slowest == 15.0 and status == "ok"
        assert value == pytest.approx(2 * 1.0e6 / 15e-3)


def test_a_failing_rank_is_seen_by_the_other():
    out, codes = _run(2, fail_rank=1)
    assert codes[1] == 3
    survivors = [o for o in out if o[0] == 0]
    assert len(survivors) == 1 and survivors[0][3] != "ok"
