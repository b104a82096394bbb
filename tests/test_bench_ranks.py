"""The benchmark's multi-process path (one replica per GPU, "replicas only": the product is
not sharded and no collective touches its data): the timed region is taken as the slowest
rank's, and the job's rate counts the work of every rank. Run here as two gloo processes on
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


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 10.0 + 5.0 * rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(elapsed, dist, torch.device("cpu"))
        rate = bench.job_rate(1000.0, world, slowest)
        results[rank] = (slowest, rate)
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_the_work():
    world = 2
    results = mp.Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), results), nprocs=world,
                       start_method="spawn")
    assert results[0] == results[1] == (15.0, 1000.0 * 2 / 0.015)


def test_single_process_is_the_identity():
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_rate(1e12, 1, 500.0) == 2e12
