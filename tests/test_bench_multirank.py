"""The multi-rank bench path on the CPU: two gloo ranks, each running its own
replica of the workload, report the max of their step times and the whole-job
throughput of both replicas (bench.py under torchrun does the same over NCCL).
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], world)
        out[rank] = (slowest, bench.replica_throughput(1000, world, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    times = [1.25, 2.5]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, times, out), nprocs=world,
                           start_method="spawn")
        results = dict(out)
    for rank in range(world):
        slowest, value = results[rank]
        assert slowest == 2.5
        assert value == pytest.approx(2 * 1000 / 2.5e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.replica_throughput(576000, 1, 0.5) == pytest.approx(576000 / 0.5e-3)
