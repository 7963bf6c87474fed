"""bench.py's step across ranks, run as two processes on cuda:0 that exchange through gloo.

A multi-GPU bench run (torchrun, NCCL) measures the layer-wise Muon step and the Sign-Muon
exchange through bench.measure and bench.run_e2e_dist. Here the same functions run with
world size 2 on one GPU: every rank runs its share of the step in the library's kernels and
gloo moves the exchanged bytes through host memory, so no kernel of one rank waits on the
other. The line must describe a strong-scaling job and both ranks must end with the same
weights.
"""

import os
import socket
import traceback

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out, config):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import bench
        from matrix_aware_optimizers_gb300 import workloads
        opts = bench.parse_args(["--config", str(config)])
        wl = workloads.workload(config)

        def barrier():
            dist.barrier()

        def max_over_ranks(x):
            return bench.reduce_max(x, dev, world)

        line, step = bench.measure(opts, wl, dev, world, rank, 0, None, 3, 3, barrier,
                                   max_over_ranks)
        e2e = bench.run_e2e_dist(step, 2, dev, barrier, max_over_ranks)
        # every rank holds the same weights after the exchange
        w = torch.cat([x.float().reshape(-1) for x in step.W])
        digest = float(w.double().abs().sum()), float(w[::997].double().sum())
        out[rank] = (line["scaling"], line["n_gpus"], line["value"] > 0, e2e["value"] > 0,
                     line["config"]["parallelism"], digest, len(step.M), None)
        dist.destroy_process_group()
    except Exception:
        out[rank] = (None,) * 7 + (traceback.format_exc(),)


@pytest.mark.parametrize("config", [2, 3])
def test_bench_step_across_two_ranks(config):
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(2, _free_port(), out, config), nprocs=2, join=True,
                       start_method="spawn")
    for r in (0, 1):
        assert out[r][7] is None, out[r][7]
        scaling, n, ok_v, ok_e, par, _, n_local, _ = out[r]
        assert scaling == "strong" and n == 2 and ok_v and ok_e
        assert ("layer-wise" if config == 2 else "split over 2 ranks") in par
    assert out[0][5] == out[1][5]  # identical weights on both ranks
    if config == 2:
        assert out[0][6] + out[1][6] == 48  # every matrix's momentum owned by one rank
    else:
        assert out[0][6] == out[1][6] == 4  # four of the eight workers per rank
