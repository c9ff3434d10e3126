"""The multi-GPU bench path is replicas with no data-path collective: each
rank times its own batch, the slowest rank's time counts, and the whole-job
throughput sums the work of all ranks.  This host logic is checked here with
two gloo ranks on the CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        my_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        m = bench.max_over_ranks(my_ms, dist, None)
        v = bench.job_throughput(1e12, world, 4, m)
        out[rank] = (m, v)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        m, v = out[rank]
        assert m == pytest.approx(15.0)
        # 2 ranks x 4 steps x 1 TFLOP in 15 ms
        assert v == pytest.approx(2 * 4 * 1.0 / 15e-3)


def test_single_process_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(2e12, 1, 10, 20.0) == pytest.approx(1000.0)
