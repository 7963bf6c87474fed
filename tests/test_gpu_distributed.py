"""The optimizer step across ranks on a GPU: two ranks (processes) on cuda:0 exchanging
through gloo, each running its share of the step in libmao's kernels.

The ranks' kernels never wait on one another: each rank's kernels finish, gloo copies the
exchanged bytes through host memory, and only then do the next kernels run. Every rank's
result must equal, bit for bit, one process stepping every matrix (Muon) or every worker
(Sign-Muon) on the same inputs:
* layer-wise Muon ([Megatron] "レイヤーごとの分散オプティマイザ", "負荷分散"): the owned
  matrices' muon_step, then the all-gather(v) of the updated weights;
* Sign-Muon ([SignMuon] §2 steps 3-4): the 1-bit all-gather of packed signs and the local
  vote, and the int8 variant's SUM all-reduce.
"""

import os
import socket
import traceback

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

QUINTIC = (3.4445, -4.7750, 2.0315)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _spawn(fn, world, *args):
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(fn, args=(world, _free_port(), out) + args, nprocs=world, join=True,
                       start_method="spawn")
    return dict(out)


def _muon_inputs(dev, shapes):
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    W = [(torch.randn(s, generator=g, device=dev) * 0.02).to(torch.bfloat16) for s in shapes]
    M = [(torch.randn(s, generator=g, device=dev) * 0.01).to(torch.bfloat16) for s in shapes]
    G = [(torch.randn(s, generator=g, device=dev) * 0.02).to(torch.bfloat16) for s in shapes]
    return W, M, G


def _layerwise_rank(rank, world, port, out):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import matrix_aware_optimizers_gb300 as mao
        from matrix_aware_optimizers_gb300 import distributed as D
        shapes = [(256, 640), (640, 256), (512, 512), (256, 1024), (384, 768), (768, 256)]
        W0, M0, G0 = _muon_inputs(dev, shapes)
        plan = D.LayerwiseMuon(shapes, torch.bfloat16, steps=5)
        flat, W = plan.layout.allocate(dev)
        for v, w in zip(W, W0):
            v.copy_(w)
        M_own = [M0[i].clone() for i in plan.mine]
        G_own = [G0[i] for i in plan.mine]
        for _ in range(2):  # two steps: the second starts from the gathered weights
            plan.step(W, M_own, G_own, 0.95, 0.02, 5, QUINTIC, flat=flat)
        torch.cuda.synchronize()
        mao.sync_status()
        # one process, every matrix, the same two steps
        Wr = [w.clone() for w in W0]
        Mr = [m.clone() for m in M0]
        for _ in range(2):
            mao.muon_step(Wr, Mr, G0, 0.95, 0.02, 5, QUINTIC)
        mao.sync_status()
        out[rank] = (all(torch.equal(a, b) for a, b in zip(W, Wr)),
                     all(torch.equal(M_own[k], Mr[i]) for k, i in enumerate(plan.mine)),
                     list(plan.mine), None)
        dist.destroy_process_group()
    except Exception:
        out[rank] = (False, False, [], traceback.format_exc())


def test_layerwise_muon_two_ranks_equal_one_process():
    out = _spawn(_layerwise_rank, 2)
    for rank in (0, 1):
        assert out[rank][3] is None, out[rank][3]
        assert out[rank][0], "rank %d weights differ from the one-process step" % rank
        assert out[rank][1], "rank %d momenta differ" % rank
    assert sorted(out[0][2] + out[1][2]) == list(range(6))
    assert out[0][2] and out[1][2]


def _sign_rank(rank, world, port, out, variant):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import matrix_aware_optimizers_gb300 as mao
        from matrix_aware_optimizers_gb300 import distributed as D
        R, C, Wn = 384, 640, 4
        g = torch.Generator(device=dev)
        g.manual_seed(12)
        W0 = (torch.randn((R, C), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        M0 = torch.randn((R, C), generator=g, device=dev).to(torch.bfloat16)
        Gs = [torch.randn((R, C), generator=g, device=dev).to(torch.bfloat16) for _ in range(Wn)]
        ex = D.SignExchange(R, C, Wn)
        mine = list(range(ex.first_worker, ex.first_worker + ex.local))
        W = W0.clone()
        M_loc = [M0.clone() for _ in mine]
        vote = torch.zeros(ex.stride, dtype=torch.int32, device=dev)
        if variant == "bits":
            words = ex.allocate_words(dev)
            D.sign_muon_step(ex, W, M_loc, [Gs[m] for m in mine], words, vote, 0.95, 1e-3, 5,
                             QUINTIC)
        else:
            U = [torch.empty((R, C), dtype=torch.bfloat16, device=dev) for _ in mine]
            s8 = torch.zeros((ex.local, ex.s_stride), dtype=torch.int8, device=dev)
            total = torch.zeros(ex.nbits, dtype=torch.int8, device=dev)
            D.sign_muon_step_int8(ex, W, M_loc, [Gs[m] for m in mine], U, s8, total, vote,
                                  0.95, 1e-3, 5, QUINTIC)
        torch.cuda.synchronize()
        mao.sync_status()
        # one process over all workers, the same calls
        Wr = W0.clone()
        Mr = [M0.clone() for _ in range(Wn)]
        mao.muon_momentum_update(Mr, Gs, 0.95)
        if variant == "bits":
            wr = torch.zeros((Wn, ex.stride), dtype=torch.int32, device=dev)
            mao.ns_orthogonalize(Mr, None, 5, QUINTIC, 1e-7, "bf16",
                                 sign_bits=[wr[m, :ex.nwords] for m in range(Wn)])
            vr = mao.majority_vote_packed(wr, ex.nbits)
            same_ex = torch.equal(words, wr)
        else:
            Ur = [torch.empty((R, C), dtype=torch.bfloat16, device=dev) for _ in range(Wn)]
            mao.ns_orthogonalize(Mr, Ur, 5, QUINTIC, 1e-7, "bf16")
            sr = torch.zeros((Wn, ex.s_stride), dtype=torch.int8, device=dev)
            for m in range(Wn):
                mao.sign_int8(Ur[m], sr[m, :ex.nbits].view(R, C))
            sums, _, vr = mao.majority_vote_int8(sr, ex.nbits, sum=True, vote=True)
            same_ex = torch.equal(total, sums)
        mao.apply_update(Wr, 1e-3, vote=vr)
        mao.sync_status()
        nw = ex.nwords
        out[rank] = (same_ex, torch.equal(vote[:nw], vr[:nw]), torch.equal(W, Wr), None)
        dist.destroy_process_group()
    except Exception:
        out[rank] = (False, False, False, traceback.format_exc())


@pytest.mark.parametrize("variant", ["bits", "int8"])
def test_sign_muon_two_ranks_equal_one_process(variant):
    out = _spawn(_sign_rank, 2, variant)
    for rank in (0, 1):
        assert out[rank][3] is None, out[rank][3]
        assert out[rank][0], "rank %d exchanged buffer differs" % rank
        assert out[rank][1], "rank %d vote differs" % rank
        assert out[rank][2], "rank %d weights differ" % rank
