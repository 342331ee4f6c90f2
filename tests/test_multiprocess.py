"""The bench's multi-rank bookkeeping on two CPU processes (gloo): the path
runs replicas (each rank the whole workload on its own inputs, no exchange),
so the job's time is the slowest rank's and its throughput counts the work of
every rank.  No GPU is involved."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        own = 10.0 + 5.0 * rank                 # this rank's timed region, ms
        ms = bench.job_ms(own, dist, torch.device("cpu"))
        units = 1.0e9                           # per rank per step
        value = bench.job_tflops(units, 4, world, ms)
        # every rank sees the same job time and value
        got = [None] * world
        dist.all_gather_object(got, (ms, value))
        out[rank] = (own, ms, value, got)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_job_time_is_max_over_ranks_and_value_counts_all_ranks(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    slowest = max(v[0] for v in res.values())
    for rank, (own, ms, value, got) in res.items():
        assert ms == slowest
        assert value == pytest.approx(1.0e9 * 4 * world / (slowest / 1e3) / 1e12)
        assert all(g == (ms, value) for g in got)


def test_single_rank_needs_no_process_group():
    assert bench.job_ms(7.5, None, None) == 7.5
    assert bench.job_tflops(2.0e12, 3, 1, 1000.0) == pytest.approx(6.0)
