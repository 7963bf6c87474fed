"""GPU parity of Newton–Schulz against the fp64 oracle.

Tolerances (relative Frobenius error of U): 1e-4 for the fp32 path, 2e-2 for the bf16
tensor-core path. Shapes span several 128 x 256 tiles, ragged tails in every
dimension, both orientations (R <= C and R > C) and grouped batches of mixed shapes.
"""

import numpy as np
import pytest
import torch

import matrix_aware_optimizers_gb300 as mao
import oracle
from helpers import bits_of, rand_matrix, rel_fro, to_np, words_np

pytestmark = pytest.mark.gpu

QUINTIC = (3.4445, -4.7750, 2.0315)
TOL = {"f32": 1e-4, "bf16": 2e-2}


def _run(ins, compute, steps=5, coeffs=QUINTIC, out_dtype=torch.float32, bits=False):
    outs = [torch.empty(x.shape, dtype=out_dtype, device=x.device) for x in ins]
    sb = [torch.full((mao.packed_words(*x.shape),), -1, dtype=torch.int32, device=x.device)
          for x in ins] if bits else None
    mao.ns_orthogonalize(ins, outs, steps=steps, coeffs=coeffs, compute=compute, sign_bits=sb)
    mao.sync_status()
    return outs, sb


@pytest.mark.parametrize("shape", [(64, 128), (128, 64), (33, 70), (70, 33), (1, 9), (9, 1),
                                   (100, 100), (130, 300)])
def test_ns_f32_parity(cuda, shape):
    gen = torch.Generator().manual_seed(21)
    X = rand_matrix(gen, shape, torch.float32, cuda)
    (U,), _ = _run([X], "f32")
    want = oracle.newton_schulz(to_np(X), 5, QUINTIC)
    assert rel_fro(to_np(U), want) <= TOL["f32"]


@pytest.mark.parametrize("shape", [(128, 256), (256, 128), (768, 768), (300, 700), (700, 300),
                                   (64, 64), (1, 40), (40, 1), (200, 1030), (1030, 200)])
def test_ns_bf16_parity(cuda, shape):
    gen = torch.Generator().manual_seed(22)
    X = rand_matrix(gen, shape, torch.bfloat16, cuda)
    (U,), _ = _run([X], "bf16")
    want = oracle.newton_schulz(to_np(X), 5, QUINTIC)
    err = rel_fro(to_np(U), want)
    assert err <= TOL["bf16"], err


@pytest.mark.parametrize("compute", ["f32", "bf16"])
def test_ns_grouped_mixed_shapes(cuda, compute):
    gen = torch.Generator().manual_seed(23)
    shapes = [(256, 768), (768, 256), (256, 256), (256, 768), (96, 200), (768, 256)]
    dt = torch.bfloat16 if compute == "bf16" else torch.float32
    Xs = [rand_matrix(gen, s, dt, cuda, 0.01 * (i + 1)) for i, s in enumerate(shapes)]
    Us, _ = _run(Xs, compute)
    for X, U in zip(Xs, Us):
        assert rel_fro(to_np(U), oracle.newton_schulz(to_np(X), 5, QUINTIC)) <= TOL[compute]


@pytest.mark.parametrize("compute", ["f32", "bf16"])
def test_ns_per_step_coefficients_and_steps(cuda, compute):
    gen = torch.Generator().manual_seed(24)
    dt = torch.bfloat16 if compute == "bf16" else torch.float32
    X = rand_matrix(gen, (192, 320), dt, cuda)
    co = [(3.0, -3.2, 1.2), (2.0, -1.5, 0.5), QUINTIC]
    (U,), _ = _run([X], compute, steps=3, coeffs=co)
    assert rel_fro(to_np(U), oracle.newton_schulz(to_np(X), 3, co)) <= TOL[compute]
    (U1,), _ = _run([X], compute, steps=1)
    assert rel_fro(to_np(U1), oracle.newton_schulz(to_np(X), 1, QUINTIC)) <= TOL[compute]


@pytest.mark.parametrize("compute", ["f32", "bf16"])
def test_ns_cubic_converges_to_polar(cuda, compute):
    gen = torch.Generator().manual_seed(25)
    dt = torch.bfloat16 if compute == "bf16" else torch.float32
    # well-conditioned input: normalised singular values spread over [0.3, 1] * scale
    rng = np.random.default_rng(5)
    Q1, _ = np.linalg.qr(rng.standard_normal((96, 96)))
    Q2, _ = np.linalg.qr(rng.standard_normal((160, 160)))
    M = (Q1 * np.linspace(1.0, 0.3, 96)) @ Q2[:, :96].T
    X = torch.from_numpy(M.astype(np.float32)).to(dt).to(cuda)
    (U,), _ = _run([X], compute, steps=40, coeffs=(1.5, -0.5, 0.0))
    want = oracle.newton_schulz(to_np(X), 40, (1.5, -0.5, 0.0))
    assert rel_fro(to_np(U), want) <= TOL[compute]


@pytest.mark.parametrize("compute", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(64, 128), (96, 200), (200, 96), (256, 512)])
def test_fused_sign_bits_match_output(cuda, compute, shape):
    # the signs written by the last product's epilogue are the signs of the fp32 U
    gen = torch.Generator().manual_seed(26)
    dt = torch.bfloat16 if compute == "bf16" else torch.float32
    X = rand_matrix(gen, shape, dt, cuda)
    (U,), (bits,) = _run([X], compute, bits=True)
    got = bits_of(words_np(bits), shape[0] * shape[1])
    assert np.array_equal(got, (to_np(U).reshape(-1) >= 0).astype(np.uint8) |
                          np.isnan(to_np(U).reshape(-1)).astype(np.uint8))
    # and sign-only requests (no U written) give the same words
    sb = [torch.zeros(mao.packed_words(*shape), dtype=torch.int32, device=cuda)]
    mao.ns_orthogonalize([X], [None], compute=compute, sign_bits=sb)
    mao.sync_status()
    assert np.array_equal(words_np(sb[0]), words_np(bits))


def test_ns_in_place_and_strided(cuda):
    gen = torch.Generator().manual_seed(27)
    X = rand_matrix(gen, (96, 200), torch.bfloat16, cuda, ld=208)
    want = oracle.newton_schulz(to_np(X), 5, QUINTIC)
    mao.ns_orthogonalize([X], [X], compute="bf16")
    mao.sync_status()
    assert rel_fro(to_np(X), want) <= TOL["bf16"]


def test_ns_zero_matrix(cuda):
    X = torch.zeros((128, 256), dtype=torch.bfloat16, device=cuda)
    (U,), (bits,) = _run([X], "bf16", bits=True)
    assert torch.count_nonzero(U).item() == 0
    assert np.all(words_np(bits) == 0xFFFFFFFF)  # +0 -> sign +1


def test_ns_output_symmetry_invariant(cuda):
    # NS(X^T) = NS(X)^T: the two orientations take different operand layouts
    gen = torch.Generator().manual_seed(28)
    X = rand_matrix(gen, (256, 640), torch.bfloat16, cuda)
    XT = X.t().contiguous()
    (U, UT), _ = _run([X, XT], "bf16")
    assert rel_fro(to_np(UT), to_np(U).T) <= 2e-2


@pytest.mark.parametrize("compute", ["f32", "bf16"])
def test_ns_more_shape_groups_than_one_launch_holds(cuda, compute):
    # eleven distinct shapes: two rounds of grouped launches (at most eight groups each)
    gen = torch.Generator().manual_seed(29)
    dt = torch.bfloat16 if compute == "bf16" else torch.float32
    shapes = [(64 + 32 * i, 96 + 48 * i) for i in range(8)] + [(300, 100), (100, 300), (256, 256)]
    Xs = [rand_matrix(gen, s, dt, cuda, 0.01 * (i + 1)) for i, s in enumerate(shapes)]
    Us, _ = _run(Xs, compute)
    for X, U in zip(Xs, Us):
        assert rel_fro(to_np(U), oracle.newton_schulz(to_np(X), 5, QUINTIC)) <= TOL[compute]
