"""The benchmark's multi-rank host logic (replicas, no data-path collective)
on two gloo ranks on the CPU: every rank contributes its step time, the job's
step time is the slowest rank's and the bytes of all ranks add up."""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_us = 100.0 + 50.0 * rank
        times = bench.max_over_ranks(my_us, world)
        value, gbps = bench.aggregate(times, [1e9] * world)
        bench.barrier(world)
        results[rank] = (times, value, gbps)
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_aggregate():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        times, value, gbps = res[rank]
        assert times == [100.0, 150.0]
        assert value == 150.0
        assert abs(gbps - 2e9 / 150e-6 / 1e9) < 1e-6
