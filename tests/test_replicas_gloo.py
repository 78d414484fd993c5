"""The multi-GPU path of bench.py is replicas only: every rank runs the same decode steps on its own GPU and the
ranks meet once, to take the slowest rank's timed time. This checks that aggregation with two gloo ranks on CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    slowest = bench.max_over_ranks(times[rank], torch.device("cpu"))
    out[rank] = (slowest, bench.whole_job_rate(20, world, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_ranks_tokens():
    world, times = 2, [1.5, 2.5]  # timed milliseconds of 20 one-token steps on each rank
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, rate = res[rank]
        assert slowest == pytest.approx(2.5)
        assert rate == pytest.approx(20 * 2 / 2.5e-3)  # tokens of both ranks over the slowest rank's time


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(3.0, torch.device("cpu")) == 3.0
    assert bench.whole_job_rate(10, 1, 2.0) == pytest.approx(5000.0)
