"""The multi-GPU path is replicas only: every rank runs the same workload on
its own GPU and the benchmark reports all ranks' work over the slowest rank's
time.  This checks that host-side reduction with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.slowest_rank_ms(10.0 + 5.0 * rank, world)  # rank 1 is slower
        out[rank] = (ms, bench.job_throughput(2e9, ms, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == pytest.approx(15.0)
    # 2 ranks x 2 GFLOP per step over 15 ms
    assert out[0][1] == pytest.approx(2 * 2e9 / 15e-3 / 1e9)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(3.5, 1) == 3.5
    assert bench.job_throughput(1e9, 1.0, 1) == pytest.approx(1000.0)
