"""Pins of the Dion oracle against facts that do not come from the oracle itself.

[Dion] (dsdanielpark.github.io), algorithm section: B = M + G, a single power iteration
warm-started from Q_prev, error-feedback momentum, ColumnNormalize, update X - lr P Q^T.
"""

import numpy as np
import pytest

import oracle


def _gram_schmidt(P):
    """Classical Gram-Schmidt with reorthogonalisation, column by column (small inputs)."""
    P = np.asarray(P, np.float64)
    m, r = P.shape
    Q = np.zeros((m, r))
    for k in range(r):
        v = P[:, k].copy()
        for _ in range(2):
            for j in range(k):
                v -= (Q[:, j] @ v) * Q[:, j]
        Q[:, k] = v / np.linalg.norm(v)
    return Q


@pytest.mark.parametrize("shape", [(8, 3), (20, 7), (64, 16), (5, 5)])
def test_orthonormalise_matches_gram_schmidt(shape):
    rng = np.random.default_rng(70 + shape[0])
    P = rng.standard_normal(shape)
    got = oracle.orthonormalise_columns(P)
    assert np.allclose(got, _gram_schmidt(P), atol=1e-10)
    assert np.allclose(got.T @ got, np.eye(shape[1]), atol=1e-12)
    # P = Q T with T upper triangular and a positive diagonal
    T = got.T @ P
    assert np.allclose(np.tril(T, -1), 0, atol=1e-10) and np.all(np.diag(T) > 0)


def test_column_normalize():
    R = np.array([[3.0, 0.0, -1.0], [4.0, 0.0, 0.0]])
    Q = oracle.column_normalize(R)
    assert np.allclose(Q, [[0.6, 0.0, -1.0], [0.8, 0.0, 0.0]])


def test_exact_low_rank_buffer_gives_polar_factor():
    # B of exact rank r and Q_prev = its right singular vectors: P = U, R = V S, Q = V, so
    # the update direction P Q^T is U V^T, the orthogonalised buffer (the Muon direction)
    rng = np.random.default_rng(71)
    m, n, r = 24, 40, 5
    U, _ = np.linalg.qr(rng.standard_normal((m, r)))
    V, _ = np.linalg.qr(rng.standard_normal((n, r)))
    S = np.diag([5.0, 3.0, 2.0, 1.0, 0.5])
    B = U @ S @ V.T
    M = 0.25 * B
    G = B - M
    X = rng.standard_normal((m, n))
    out = oracle.dion_step(X, M, G, V, mu=0.9, lr=0.1)
    assert np.allclose(out["P"] @ out["Q"].T, U @ V.T, atol=1e-10)
    assert np.allclose(out["X"], X - 0.1 * U @ V.T, atol=1e-10)
    # the rank-r component is removed up to the momentum share: M = mu B
    assert np.allclose(out["M"], 0.9 * B, atol=1e-10)


@pytest.mark.parametrize("m,n", [(6, 10), (10, 6)])
def test_full_rank_keeps_mu_times_buffer(m, n):
    rng = np.random.default_rng(72 + m)
    r = min(m, n)
    M, G = rng.standard_normal((m, n)), rng.standard_normal((m, n))
    Q0 = rng.standard_normal((n, r))
    out = oracle.dion_step(np.zeros((m, n)), M, G, Q0, mu=0.95, lr=1.0)
    # with r = min(m, n) and an invertible start, span(P) is the column space of B, so
    # the projection keeps all of B and only the momentum share remains
    assert np.allclose(out["M"], 0.95 * (M + G), atol=1e-10)


def test_error_feedback_identity_and_projection():
    rng = np.random.default_rng(73)
    m, n, r = 30, 50, 6
    M, G = rng.standard_normal((m, n)), rng.standard_normal((m, n))
    Q0 = rng.standard_normal((n, r))
    out = oracle.dion_step(np.zeros((m, n)), M, G, Q0, mu=0.8, lr=1.0)
    B = M + G
    assert np.allclose(out["M"] + 0.2 * out["P"] @ out["R"].T, B, atol=1e-10)
    assert np.allclose(out["P"] @ out["R"].T, out["P"] @ out["P"].T @ B, atol=1e-10)
    # the direction's columns: Q has unit columns and P orthonormal ones
    assert np.allclose(np.linalg.norm(out["Q"], axis=0), 1.0)
    assert np.allclose(out["P"].T @ out["P"], np.eye(r), atol=1e-12)


def test_warm_start_converges_to_top_subspace():
    # repeated steps on a fixed buffer are repeated power iterations: span(P) approaches
    # the top-r left singular subspace of B
    rng = np.random.default_rng(74)
    m, n, r = 20, 30, 3
    B = rng.standard_normal((m, n)) @ np.diag(np.linspace(3, 0.1, n)) @ rng.standard_normal((n, n))
    U = np.linalg.svd(B)[0][:, :r]
    Q = rng.standard_normal((n, r))
    for _ in range(60):
        out = oracle.dion_step(np.zeros((m, n)), np.zeros((m, n)), B, Q, mu=0.5, lr=0.0)
        Q = out["Q"]
    proj = out["P"] @ out["P"].T
    assert np.linalg.norm(proj @ U - U) < 1e-6
