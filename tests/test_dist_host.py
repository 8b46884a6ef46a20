"""The multi-rank host logic of bench.py on CPU: two ranks over gloo (one
process per GPU on a GPU node, here plain processes).  The ranks are
independent replicas of the layer; the process group carries only the barrier
around the timed region and the max over ranks of its duration, and the
reported value is the units of all ranks over the slowest rank's time."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(world, backend="gloo")
    bench.barrier(w)
    mx = bench.allreduce_max(w, 1.0 + r)            # rank r timed 1 + r seconds
    value, total = bench.job_throughput(w, 100.0, 1.0 + r)
    bench.barrier(w)
    dist.destroy_process_group()
    out.put((r, w, mx, value, total))


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_report_the_slowest_rank_and_the_whole_job(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, mx, value, total in res:
        assert w == world
        assert mx == float(world) and total == float(world)  # the slowest rank
        assert value == pytest.approx(100.0 * world / world)  # all ranks' units over that time


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.allreduce_max(1, 2.5) == 2.5
    assert bench.job_throughput(1, 10.0, 2.0) == (5.0, 2.0)
