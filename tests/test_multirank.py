"""The bench's multi-rank host logic (replicas: one process per GPU, no data
exchange) on CPU with the gloo backend, world size 2: the job time is the
slowest rank's and the whole-job value counts every rank's work."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        job_ms = bench.max_over_ranks(ms, world, torch.device("cpu"))
        value = bench.replica_throughput(1e12, 4, job_ms, world)
        out[rank] = (job_ms, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        ctx = mp.get_context("spawn")
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    # every rank sees the slowest rank's time; the value counts both ranks' work
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == pytest.approx(2 * 1e12 * 4 / 15e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.replica_throughput(1e12, 2, 1.0, 1) == pytest.approx(2000.0)
