"""The optimizer step across ranks, on CPU: the owner plan, and the exchanges as two gloo
ranks (world size 2) run them.

* Layer-wise Muon ([Megatron] "レイヤーごとの分散オプティマイザ", "負荷分散"): whole matrices
  per rank, chosen by Newton–Schulz flops, then one all-gather(v) of the updated weights.
* Sign-Muon ([SignMuon] §2 "Fluxo Algorítmico (Distribuído)", steps 3-4): packed signs
  all-gathered into every rank's own [W_n][stride] buffer, then the local vote; the int8
  variant's SUM all-reduce.

The ranks' local stages are computed here by the fp64 oracle (these tests have no GPU); the
exchange is the package's code. Every rank's result must equal, bit for bit, the oracle's
single-process step over all matrices or all workers.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from matrix_aware_optimizers_gb300 import distributed as D
from matrix_aware_optimizers_gb300 import workloads

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
    port = _free_port()
    mp.start_processes(fn, args=(world, port, out) + args, nprocs=world, join=True,
                       start_method="spawn")
    return dict(out)


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


# ------------------------------------------------------------------ owner plan

@pytest.mark.parametrize("index", [4, 5, 2])
@pytest.mark.parametrize("world", [2, 4, 8])
def test_lpt_plan_balances_ns_flops(index, world):
    shapes = workloads.workload(index).shapes
    costs = [D.ns_flops(R, C, 5) for R, C in shapes]
    owners, loads = D.assign_lpt(costs, world)
    assert sorted(set(owners)) == list(range(world))
    # every matrix on exactly one rank, and the loads are the sums of the owned costs
    for r in range(world):
        assert loads[r] == sum(c for c, o in zip(costs, owners) if o == r)
    assert sum(loads) == sum(costs)
    mean = sum(costs) / world
    # LPT bound: max load <= mean + largest unit; on these shape lists it is within 3%
    assert max(loads) <= mean + max(costs)
    assert max(loads) / mean <= 1.03, max(loads) / mean
    rr = D.assign_round_robin(len(costs), world)
    rr_loads = [sum(c for c, o in zip(costs, rr) if o == r) for r in range(world)]
    assert max(loads) <= max(rr_loads)
    # the same plan on every rank: a pure function of the shapes
    assert D.assign_lpt(costs, world) == (owners, loads)


def test_lpt_plan_beats_round_robin_on_moe_experts():
    # 385 matrices: 128 experts x (2048x768, 2048x768, 768x2048) + one 2048x2048 block;
    # round-robin over 3 ranks puts every expert's first matrix on rank 0, ... and the
    # dense block on one of them; the cost model evens the loads
    shapes = workloads.workload(5).shapes
    costs = [D.ns_flops(R, C, 5) for R, C in shapes]
    _, loads = D.assign_lpt(costs, 8)
    rr = D.assign_round_robin(len(costs), 8)
    rr_loads = [sum(c for c, o in zip(costs, rr) if o == r) for r in range(8)]
    assert max(loads) < max(rr_loads)


def test_ns_flops_is_the_dense_count():
    assert D.ns_flops(64, 128, 5) == oracle.ns_dense_flops(64, 128, 5)
    assert D.ns_flops(14336, 4096, 5) == oracle.ns_dense_flops(4096, 14336, 5)


def test_weight_layout_segments():
    shapes = [(4, 6), (3, 5), (8, 8), (2, 2)]
    owners = [1, 0, 0, 1]
    lay = D.WeightLayout(shapes, torch.float32, owners, 2)
    flat, views = lay.allocate("cpu")
    assert flat.numel() == 2 * lay.segment_bytes
    for i, v in enumerate(views):
        assert tuple(v.shape) == shapes[i]
        start = v.data_ptr() - flat.data_ptr()
        assert start % D.SEGMENT_ALIGN == 0
        assert owners[i] * lay.segment_bytes <= start < (owners[i] + 1) * lay.segment_bytes
    # views do not overlap
    spans = sorted((v.data_ptr(), v.data_ptr() + v.numel() * 4) for v in views)
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))


# ------------------------------------------------------------------ layer-wise Muon

def _muon_case():
    rng = np.random.default_rng(5)
    shapes = [(24, 40), (40, 24), (32, 32), (16, 48), (48, 16), (8, 64), (20, 20)]
    W = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    M = [oracle.bf16_rne((rng.standard_normal(s) * 0.01).astype(np.float32)) for s in shapes]
    G = [oracle.bf16_rne((rng.standard_normal(s) * 0.02).astype(np.float32)) for s in shapes]
    return shapes, W, M, G


def _layerwise_rank(rank, world, port, out):
    _init(rank, world, port)
    try:
        shapes, W, M, G = _muon_case()
        plan = D.LayerwiseMuon(shapes, w_dtype=torch.float64, steps=5)
        assert plan.world == world and plan.rank == rank
        flat, views = plan.layout.allocate("cpu")
        # local stage of this rank: the owned matrices only (the oracle stands in for the
        # CUDA step here); other ranks' views stay zero until the all-gather
        for i in plan.mine:
            r = oracle.muon_step([W[i]], [M[i]], [G[i]], 0.95, 0.02, 5, QUINTIC, m_store="bf16")
            views[i].copy_(torch.from_numpy(r["W"][0]))
        D.allgather_weights(plan.layout, flat)
        out[rank] = ([v.numpy().copy() for v in views], plan.mine)
    finally:
        dist.destroy_process_group()


def test_layerwise_muon_two_gloo_ranks_equal_single_process():
    out = _spawn(_layerwise_rank, 2)
    shapes, W, M, G = _muon_case()
    ref = oracle.muon_step(W, M, G, 0.95, 0.02, 5, QUINTIC, m_store="bf16")["W"]
    owned = sorted(out[0][1] + out[1][1])
    assert owned == list(range(len(shapes)))          # every matrix owned exactly once
    assert out[0][1] and out[1][1]                     # both ranks have work
    for rank in (0, 1):
        for i, w in enumerate(out[rank][0]):
            assert np.array_equal(w, ref[i]), (rank, i)


# ------------------------------------------------------------------ Sign-Muon

def _sign_case(Wn=4, R=12, C=20):
    rng = np.random.default_rng(6)
    W = oracle.bf16_rne((rng.standard_normal((R, C)) * 0.02).astype(np.float32))
    M0 = oracle.bf16_rne(rng.standard_normal((R, C)).astype(np.float32))
    Ms = [M0.copy() for _ in range(Wn)]
    Gs = [oracle.bf16_rne(rng.standard_normal((R, C)).astype(np.float32)) for _ in range(Wn)]
    return W, Ms, Gs


def _sign_rank(rank, world, port, out, variant):
    _init(rank, world, port)
    try:
        W, Ms, Gs = _sign_case()
        R, C = W.shape
        ex = D.SignExchange(R, C, len(Ms))
        w0 = ex.first_worker
        if variant == "bits":
            words = ex.allocate_words("cpu")
            for k, row in enumerate(ex.my_words(words)):
                m = w0 + k
                Mm = oracle.momentum(Ms[m], Gs[m], 0.95, "bf16")
                S = oracle.sign_of(oracle.newton_schulz(Mm, 5, QUINTIC))
                row.copy_(torch.from_numpy(oracle.pack_signs(S).view(np.int32)))
            ex.allgather_words(words)
            w = words[:, :ex.nwords].numpy().view(np.uint32)
            vote = oracle.majority_vote(w, ex.nbits)
            out[rank] = (w.copy(), vote)
        else:
            total = torch.zeros(ex.nbits, dtype=torch.int8)
            for k in range(ex.local):
                m = w0 + k
                Mm = oracle.momentum(Ms[m], Gs[m], 0.95, "bf16")
                total += torch.from_numpy(oracle.sign_of(oracle.newton_schulz(Mm, 5, QUINTIC)).reshape(-1))
            ex.allreduce_int8(total)
            s = total.numpy().astype(np.int64)
            out[rank] = (s.copy(), np.where(s >= 0, 1, -1).astype(np.int8))
    finally:
        dist.destroy_process_group()


def test_sign_muon_allgather_two_gloo_ranks_equal_single_process():
    out = _spawn(_sign_rank, 2, "bits")
    W, Ms, Gs = _sign_case()
    ref = oracle.sign_muon_step(W, Ms, Gs, 0.95, 1e-3, 5, QUINTIC, m_store="bf16", w_store="bf16")
    for rank in (0, 1):
        words, vote = out[rank]
        assert np.array_equal(words, ref["words"]), rank   # [W_n][nwords], every worker's row
        assert np.array_equal(vote, ref["vote"]), rank


def test_sign_muon_int8_allreduce_two_gloo_ranks_equal_single_process():
    out = _spawn(_sign_rank, 2, "int8")
    W, Ms, Gs = _sign_case()
    ref = oracle.sign_muon_step(W, Ms, Gs, 0.95, 1e-3, 5, QUINTIC, m_store="bf16", w_store="bf16",
                                variant="int8")
    for rank in (0, 1):
        sums, s_bar = out[rank]
        assert np.array_equal(sums, ref["sums"].reshape(-1)), rank
        assert np.array_equal(s_bar, ref["S_bar"].reshape(-1)), rank


def test_sign_exchange_rejects_uneven_split_and_int8_overflow():
    ex = D.SignExchange(4, 4, 3)  # world 1: any worker count
    assert ex.local == 3 and ex.first_worker == 0
    with pytest.raises(ValueError):
        D.SignExchange(4, 4, 200).allreduce_int8(torch.zeros(16, dtype=torch.int8))
