"""GPU parity of the HBM-bound stages against the oracle: bit-exact.

momentum, sign + pack, majority vote and update have unique results on identical
inputs, so the CUDA path must reproduce the oracle's bits exactly.
"""

import numpy as np
import pytest
import torch

import matrix_aware_optimizers_gb300 as mao
import oracle
from helpers import bits_of, rand_matrix, to_np, words_np

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.mark.parametrize("mdt,gdt", [("bf16", "bf16"), ("f32", "f32"), ("f32", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("shape,ld", [((64, 128), None), ((7, 13), None), ((33, 96), 104),
                                      ((1, 1), None), ((300, 1000), None)])
def test_momentum_bit_exact(cuda, mdt, gdt, shape, ld):
    gen = torch.Generator().manual_seed(11)
    M = rand_matrix(gen, shape, DT[mdt], cuda, 1.0, ld)
    G = rand_matrix(gen, shape, DT[gdt], cuda, 0.5, ld)
    want = oracle.momentum(to_np(M), to_np(G), 0.95, mdt)
    mao.muon_momentum_update(M, G, 0.95)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(M).view(np.uint32), want.view(np.uint32))


def test_momentum_grouped_batch(cuda):
    gen = torch.Generator().manual_seed(12)
    shapes = [(768, 2304), (768, 768), (33, 7), (3072, 768)]
    Ms = [rand_matrix(gen, s, torch.bfloat16, cuda, 0.01) for s in shapes]
    Gs = [rand_matrix(gen, s, torch.bfloat16, cuda, 0.02) for s in shapes]
    want = [oracle.momentum(to_np(m), to_np(g), 0.95, "bf16") for m, g in zip(Ms, Gs)]
    mao.muon_momentum_update(Ms, Gs, 0.95)
    torch.cuda.synchronize()
    for m, w in zip(Ms, want):
        assert np.array_equal(to_np(m), w)


def _special_values(gen, shape, dtype, device):
    U = torch.randn(shape, generator=gen)
    flat = U.view(-1)
    n = flat.numel()
    idx = torch.randperm(n, generator=gen)
    flat[idx[: n // 10]] = 0.0
    flat[idx[n // 10: n // 5]] = -0.0
    if n >= 20:
        flat[idx[n // 5]] = float("nan")
        flat[idx[n // 5 + 1]] = -float("inf")
        flat[idx[n // 5 + 2]] = 1e-40
        flat[idx[n // 5 + 3]] = -1e-40
    return U.to(dtype).to(device)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 8), (7, 13), (64, 128), (33, 96), (4096, 64), (5, 1000)])
def test_sign_pack_bit_exact(cuda, dt, shape):
    gen = torch.Generator().manual_seed(13)
    U = _special_values(gen, shape, DT[dt], cuda)
    bits = mao.sign_pack_bits(U)
    torch.cuda.synchronize()
    want = oracle.pack_signs(oracle.sign_of(to_np(U)))
    assert np.array_equal(words_np(bits), want)


def test_sign_pack_strided(cuda):
    gen = torch.Generator().manual_seed(14)
    U = rand_matrix(gen, (40, 64), torch.bfloat16, cuda, 1.0, ld=72)
    bits = mao.sign_pack_bits(U)
    torch.cuda.synchronize()
    assert np.array_equal(words_np(bits), oracle.pack_signs(oracle.sign_of(to_np(U))))


@pytest.mark.parametrize("Wn", [1, 2, 3, 4, 7, 8, 15, 16, 33, 255, 256, 300])
@pytest.mark.parametrize("nbits", [1, 31, 32, 100, 4096, 1000003])
def test_vote_bit_exact(cuda, Wn, nbits):
    rng = np.random.default_rng(Wn * 1000 + nbits % 1000)
    nw = (nbits + 31) // 32
    stride = nw + (4 - nw % 4) % 4 if Wn % 2 else nw
    words = np.zeros((Wn, stride), np.uint32)
    words[:, :nw] = rng.integers(0, 2 ** 32, (Wn, nw), dtype=np.uint64).astype(np.uint32)
    if nbits % 32:
        words[:, nw - 1] &= np.uint32((1 << (nbits % 32)) - 1)  # padding bits are 0
    bits = torch.from_numpy(words.view(np.int32)).to(cuda)
    vote = mao.majority_vote_packed(bits, nbits)
    torch.cuda.synchronize()
    want = oracle.majority_vote(words[:, :nw], nbits)
    assert np.array_equal(words_np(vote), want)


def test_vote_all_tie_patterns(cuda):
    # exhaustive: every pattern of 8 workers at one entry (ties give +1)
    import itertools
    pats = np.array(list(itertools.product([0, 1], repeat=8)), np.uint8)  # [256][8]
    words = np.stack([np.packbits(pats[:, m], bitorder="little").view("<u4") for m in range(8)])
    bits = torch.from_numpy(words.astype(np.uint32).view(np.int32)).to(cuda)
    vote = words_np(mao.majority_vote_packed(bits, 256))
    got = bits_of(vote, 256)
    assert np.array_equal(got, (2 * pats.sum(1) >= 8).astype(np.uint8))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(64, 128), (7, 13), (33, 96), (512, 520)])
def test_update_sign_bit_exact(cuda, dt, shape):
    gen = torch.Generator().manual_seed(15)
    W = rand_matrix(gen, shape, DT[dt], cuda, 0.02)
    S = np.where(np.random.default_rng(3).random(shape) < 0.5, -1, 1).astype(np.int8)
    vote = torch.from_numpy(oracle.pack_signs(S).view(np.int32)).to(cuda)
    want = oracle.apply_update(to_np(W), S, 1e-3, dt)
    mao.apply_update(W, 1e-3, vote=vote)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(W), want)


@pytest.mark.parametrize("wdt,udt", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32")])
@pytest.mark.parametrize("shape,ld", [((64, 128), None), ((7, 13), None), ((96, 40), 48)])
def test_update_muon_bit_exact(cuda, wdt, udt, shape, ld):
    gen = torch.Generator().manual_seed(16)
    W = rand_matrix(gen, shape, DT[wdt], cuda, 0.02, ld)
    U = rand_matrix(gen, shape, DT[udt], cuda, 1.0)
    want = oracle.apply_update(to_np(W), to_np(U), 0.02, wdt)
    mao.apply_update(W, 0.02, U=U)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(W), want)


def test_update_hand_table_on_gpu(cuda, golden_dir):
    import os
    rows = []
    with open(os.path.join(golden_dir, "update_rounding.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    W = torch.tensor([[float(r[0]) for r in rows]], dtype=torch.bfloat16, device=cuda)
    S = np.array([[int(r[1]) for r in rows]], np.int8)
    vote = torch.from_numpy(oracle.pack_signs(S).view(np.int32)).to(cuda)
    mao.apply_update(W, 1e-3, vote=vote)
    torch.cuda.synchronize()
    assert to_np(W)[0].tolist() == [float(r[2]) for r in rows]
