"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks, each with its
own replica of the work (weak scaling), combine into the slowest rank's step
time and the sum of all ranks' bytes."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms, total = bench.combine_ranks(1.5 + rank, 1000 + 10 * rank, dist, "cpu")
        results[rank] = (ms, total)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_bytes():
    world = 2
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    for r in range(world):
        assert results[r] == (2.5, 2010)


def test_single_process_passes_values_through():
    import bench
    assert bench.combine_ranks(3.0, 77) == (3.0, 77)
