"""bench.py's rank aggregation on CPU: two gloo ranks (world size 2).

Every rank times its own steps; the job's time is the slowest rank's (max over ranks).
With strong scaling (a Muon or Sign-Muon step split over the ranks) the ranks together
take K steps in that time; with weak scaling (Dion replicas) every rank takes K steps.
The data-path exchanges themselves are tested in test_distributed_cpu.py.
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
        out[rank] = (ms, bench.job_throughput(ms, 10, world, "weak"),
                     bench.job_throughput(ms, 10, world, "strong"))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_steps():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == 150.0
    # weak: 2 ranks x 10 steps in the slowest rank's 150 ms; strong: 10 steps of the job
    assert out[0][1] == pytest.approx(2 * 10 / 0.150)
    assert out[0][2] == pytest.approx(10 / 0.150)


def test_single_rank_is_identity():
    assert bench.reduce_max(3.5, "cpu", 1) == 3.5
    assert bench.job_throughput(100.0, 5, 1) == pytest.approx(50.0)


def test_scaling_kinds():
    from matrix_aware_optimizers_gb300 import workloads
    assert bench.scaling_of(workloads.workload(2), 8) == "strong"
    assert bench.scaling_of(workloads.workload(3), 8) == "strong"
    assert bench.scaling_of(workloads.workload(6), 8) == "weak"
    assert bench.scaling_of(workloads.workload(6), 1) == "strong"
