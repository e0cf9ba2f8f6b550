"""The multi-GPU form of the path is replicas only (no exchange step): the
bench's max-over-ranks timing and whole-job rate, run as two gloo ranks on
the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow replica
        slowest = bench.reduce_max(ms, dist, "cpu")
        rate = bench.whole_job_rate(1000.0, world, slowest * 1e-3)
        out[rank] = (slowest, rate)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        slowest, rate = res[r]
        assert slowest == pytest.approx(15.0)
        assert rate == pytest.approx(2 * 1000.0 / 0.015)


def test_single_process_is_identity():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
