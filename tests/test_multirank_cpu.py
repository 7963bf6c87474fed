"""The multi-rank path of bench.py on CPU: two gloo ranks (world size 2).

Each rank of a multi-GPU run steps its own copy of the workload (the matrices of a
Muon step are independent units), so the only cross-rank traffic is the barrier and
the max of the timings; the job throughput counts every rank's steps over the slowest
rank's time. No data-path collective exists to test.
"""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 150.0][rank]
        dist.barrier()
        ms = bench.reduce_max(local_ms, "cpu", world)
        out[rank] = (ms, bench.job_throughput(ms, 10, world))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_steps():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == 150.0
    # 2 ranks x 10 steps in the slowest rank's 150 ms
    assert out[0][1] == pytest.approx(2 * 10 / 0.150)


def test_single_rank_is_identity():
    assert bench.reduce_max(3.5, "cpu", 1) == 3.5
    assert bench.job_throughput(100.0, 5, 1) == pytest.approx(50.0)
