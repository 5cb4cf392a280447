"""bench.py's multi-rank bookkeeping, on CPU: two ranks over gloo.

The path does not shard (one GPU holds the whole cube), so N ranks run N
independent replicas: the job's time is the slowest rank's, its throughput
counts every rank's work, and only rank 0 reports (in the reference arm,
the other ranks return without work)."""
import contextlib
import io
import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total = bench.slowest_rank_ms(10.0 + 5.0 * rank, world, dist, "cpu")
        value = bench.job_value(world, 2.0e9, 4, total, 1e12)
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            ran = bench.run_reference(types.SimpleNamespace(workload="layer_q2"), rank) if rank != 0 else None
        q.put((rank, total, value, out.getvalue(), ran))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_all_work():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, value, printed, ran in res:
        assert total == 15.0                       # rank 1's 15 ms, seen by both ranks
        assert value == pytest.approx(2 * 2.0e9 * 4 / 0.015 / 1e12)
        if rank == 1:
            assert printed == "" and ran is None   # the reference arm: nothing on rank 1


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(12.5, 1, None, "cpu") == 12.5
    assert bench.job_value(1, 1.0e9, 2, 1000.0, 1e9) == pytest.approx(2.0)
