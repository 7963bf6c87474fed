"""GPU parity of one Dion step against the fp64 oracle ([Dion], algorithm section).

The dense products take bf16 operands with fp32 accumulation, so every output is checked
with the bf16 bound used for Newton–Schulz: relative Frobenius error <= 2e-2 of
  * P (the orthonormal basis; both sides use the QR convention with a positive diagonal),
  * Q (the new, column-normalised right factor),
  * the momentum correction B - M_new = (1 - mu) P R^T,
  * the parameter change X_prev - X_new = lr P Q^T.
Closed forms checked on the GPU alone: P has orthonormal columns, Q unit columns, and an
exact rank-r buffer with Q_prev = its right singular vectors gives the update U V^T.
"""

import numpy as np
import pytest
import torch

import matrix_aware_optimizers_gb300 as mao
import oracle
from helpers import rel_fro, to_np

pytestmark = pytest.mark.gpu

TOL = 2e-2
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _inputs(gen, m, n, r, mdt, xdt, dev, gscale=1.0):
    M = (torch.randn((m, n), generator=gen) * 0.5).to(DT[mdt]).to(dev)
    G = (torch.randn((m, n), generator=gen) * gscale).to(DT[mdt]).to(dev)
    X = (torch.randn((m, n), generator=gen)).to(DT[xdt]).to(dev)
    Q = torch.randn((n, r), generator=gen).to(dev)
    Q = Q / Q.norm(dim=0, keepdim=True)
    return X, M, G, Q


def _check(out, host, X, M, Q, P, mu, lr):
    X0, M0, G0, Q0 = host
    B = M0.astype(np.float64) + G0
    assert rel_fro(to_np(P), out["P"]) <= TOL
    assert np.allclose(to_np(P).T @ to_np(P), np.eye(P.shape[1]), atol=2e-3)
    assert rel_fro(to_np(Q), out["Q"]) <= TOL
    assert np.allclose(np.linalg.norm(to_np(Q), axis=0), 1.0, atol=1e-4)
    # momentum: the correction within TOL, plus the two roundings to M's storage type
    # (B = M + G is stored, then M_new), each at most eps |value| per element
    eps = 2.0 ** -8 if M.dtype == torch.bfloat16 else 2.0 ** -24  # unit roundoff
    err = np.linalg.norm(to_np(M) - out["M"])
    assert err <= TOL * np.linalg.norm(B - out["M"]) + 2 * eps * np.linalg.norm(out["M"]) \
        + eps * np.linalg.norm(B)
    assert rel_fro(X0 - to_np(X), X0 - out["X"]) <= TOL


@pytest.mark.parametrize("m,n,r", [(256, 640, 32), (768, 768, 192), (300, 1000, 48),
                                   (1000, 300, 64), (768, 3072, 192), (200, 72, 16),
                                   (512, 768, 256), (400, 640, 200), (300, 300, 1),
                                   (96, 20, 8), (20, 96, 8)])
@pytest.mark.parametrize("mdt,xdt", [("f32", "f32"), ("bf16", "f32")])
def test_dion_step_parity(cuda, m, n, r, mdt, xdt):
    gen = torch.Generator().manual_seed(80 + m + r)
    X, M, G, Q = _inputs(gen, m, n, r, mdt, xdt, cuda)
    host = [to_np(t) for t in (X, M, G, Q)]
    P = torch.empty((m, r), dtype=torch.float32, device=cuda)
    mao.dion_step(X, M, G, Q, mu=0.95, lr=0.5, P_out=P)
    mao.sync_status()
    out = oracle.dion_step(*host, mu=0.95, lr=0.5)
    _check(out, host, X, M, Q, P, 0.95, 0.5)


def test_dion_bf16_parameters(cuda):
    # bf16 X and M
    gen = torch.Generator().manual_seed(81)
    X, M, G, Q = _inputs(gen, 512, 768, 64, "bf16", "bf16", cuda)
    host = [to_np(t) for t in (X, M, G, Q)]
    mao.dion_step(X, M, G, Q, mu=0.9, lr=1.0)
    mao.sync_status()
    out = oracle.dion_step(*host, mu=0.9, lr=1.0)
    # the change within TOL, plus the one rounding of X_new to bf16 (eps |X_new| per element)
    err = np.linalg.norm(to_np(X) - out["X"])
    assert err <= TOL * np.linalg.norm(host[0] - out["X"]) + 2.0 ** -8 * np.linalg.norm(out["X"])


def test_dion_batch_and_mixed_shapes(cuda):
    gen = torch.Generator().manual_seed(82)
    shapes = [(256, 768, 64), (256, 768, 64), (768, 256, 64), (384, 384, 64), (256, 768, 64),
              (520, 1000, 64)]
    sets = [_inputs(gen, m, n, r, "bf16", "f32", cuda) for m, n, r in shapes]
    hosts = [[to_np(t) for t in s] for s in sets]
    Ps = [torch.empty((m, r), dtype=torch.float32, device=cuda) for m, n, r in shapes]
    mao.dion_step([s[0] for s in sets], [s[1] for s in sets], [s[2] for s in sets],
                  [s[3] for s in sets], mu=0.95, lr=0.3, P_out=Ps)
    mao.sync_status()
    for s, h, P in zip(sets, hosts, Ps):
        _check(oracle.dion_step(*h, mu=0.95, lr=0.3), h, s[0], s[1], s[3], P, 0.95, 0.3)


def test_dion_deep_and_shallow_groups(cuda):
    # groups of 2048-row matrices next to 256- and 300-row ones: products of very different
    # depths in each launch (tiles dealt deepest first)
    gen = torch.Generator().manual_seed(86)
    shapes = [(256, 512, 32), (2048, 512, 32), (2048, 512, 32), (300, 700, 32)]
    sets = [_inputs(gen, m, n, r, "bf16", "f32", cuda) for m, n, r in shapes]
    hosts = [[to_np(t) for t in s] for s in sets]
    Ps = [torch.empty((m, r), dtype=torch.float32, device=cuda) for m, n, r in shapes]
    mao.dion_step([s[0] for s in sets], [s[1] for s in sets], [s[2] for s in sets],
                  [s[3] for s in sets], mu=0.95, lr=0.3, P_out=Ps)
    mao.sync_status()
    for s, h, P in zip(sets, hosts, Ps):
        _check(oracle.dion_step(*h, mu=0.95, lr=0.3), h, s[0], s[1], s[3], P, 0.95, 0.3)


def test_dion_two_steps_warm_start(cuda):
    gen = torch.Generator().manual_seed(83)
    X, M, G, Q = _inputs(gen, 512, 1024, 128, "f32", "f32", cuda)
    G2 = torch.randn((512, 1024), generator=gen).to(cuda)
    host = [to_np(t) for t in (X, M, G, Q)]
    mao.dion_step(X, M, G, Q, mu=0.9, lr=0.2)
    mao.dion_step(X, M, G2, Q, mu=0.9, lr=0.2)
    mao.sync_status()
    o1 = oracle.dion_step(*host, mu=0.9, lr=0.2)
    o2 = oracle.dion_step(o1["X"], o1["M"], to_np(G2), o1["Q"], mu=0.9, lr=0.2)
    assert rel_fro(to_np(Q), o2["Q"]) <= TOL
    assert rel_fro(host[0] - to_np(X), host[0] - o2["X"]) <= TOL


def test_dion_exact_low_rank_gives_polar_factor(cuda):
    # independent of the oracle: B = U S V^T of rank r and Q_prev = V, so the step moves X
    # by -lr U V^T and leaves M = mu B
    gen = torch.Generator().manual_seed(84)
    m, n, r = 512, 768, 32
    U = torch.linalg.qr(torch.randn((m, r), generator=gen, dtype=torch.float64))[0]
    V = torch.linalg.qr(torch.randn((n, r), generator=gen, dtype=torch.float64))[0]
    S = torch.linspace(4.0, 0.5, r, dtype=torch.float64)
    B = (U * S) @ V.T
    M = torch.zeros((m, n), dtype=torch.float32, device=cuda)
    G = B.float().to(cuda)
    X = torch.zeros((m, n), dtype=torch.float32, device=cuda)
    Q = V.float().to(cuda).contiguous()
    mao.dion_step(X, M, G, Q, mu=0.8, lr=1.0)
    mao.sync_status()
    want = -(U @ V.T).numpy()
    assert rel_fro(to_np(X), want) <= TOL
    assert rel_fro(to_np(M), 0.8 * G.double().cpu().numpy()) <= TOL


@pytest.mark.parametrize("m,n,r", [(768, 1024, 64), (3072, 768, 192), (300, 500, 40)])
def test_dion_basis_orthonormal_when_ill_conditioned(cuda, m, n, r):
    # independent of the oracle: B Q_prev with singular values spread over three decades
    # (kappa about 1e3, so one Cholesky QR pass leaves an error near kappa^2 times the
    # Gram's): after the two passes the fp32 copy of P is orthonormal to about 2^-17 (the
    # bf16-part products), checked at 2e-4, ten times tighter than the parity test's bound
    gen = torch.Generator().manual_seed(85 + r)
    U = torch.linalg.qr(torch.randn((m, r), generator=gen, dtype=torch.float64))[0]
    V = torch.linalg.qr(torch.randn((n, r), generator=gen, dtype=torch.float64))[0]
    S = torch.logspace(0.0, -3.0, r, dtype=torch.float64)
    G = ((U * S) @ V.T).float().to(cuda)
    M = torch.zeros((m, n), dtype=torch.float32, device=cuda)
    X = torch.zeros((m, n), dtype=torch.float32, device=cuda)
    Qp = V + 0.05 * torch.randn((n, r), generator=gen, dtype=torch.float64) / n ** 0.5
    Q = (Qp / Qp.norm(dim=0, keepdim=True)).float().to(cuda).contiguous()
    P = torch.empty((m, r), dtype=torch.float32, device=cuda)
    mao.dion_step(X, M, G, Q, mu=0.9, lr=0.1, P_out=P)
    mao.sync_status()
    Pd = P.double().cpu()
    assert (Pd.T @ Pd - torch.eye(r, dtype=torch.float64)).abs().max().item() <= 2e-4
    # the basis contains the leading half of B's left singular space (the trailing
    # directions, down to 1e-3 of the largest, are within the bf16 rounding of B Q_prev)
    C = Pd.T @ U[:, : r // 2]
    assert (C.T @ C - torch.eye(r // 2, dtype=torch.float64)).abs().max().item() <= 1e-2


def test_dion_zero_buffer_reports_numeric_error(cuda):
    # B = 0: B Q has no column rank, the Cholesky pivot is zero; the step leaves X and M
    # at zero and mao_sync_status reports MAO_ERR_NUMERIC (no device fault)
    m, n, r = 128, 256, 8
    X = torch.zeros((m, n), device=cuda)
    M = torch.zeros((m, n), device=cuda)
    G = torch.zeros((m, n), device=cuda)
    Q = torch.randn((n, r), device=cuda)
    mao.dion_step(X, M, G, Q, mu=0.9, lr=1.0)
    with pytest.raises(mao.MaoError) as e:
        mao.sync_status()
    assert e.value.status == 7
    mao.sync_status()  # cleared
    assert torch.count_nonzero(X) == 0 and torch.count_nonzero(M) == 0
    assert torch.isfinite(Q).all()


def test_dion_rejects_bad_arguments(cuda):
    X = torch.zeros((64, 96), device=cuda)
    Q = torch.zeros((96, 8), device=cuda)
    with pytest.raises((mao.MaoError, ValueError)):  # rank above min(m, n)
        mao.dion_step(X, X.clone(), X.clone(), torch.zeros((96, 97), device=cuda), 0.9, 1.0)
    with pytest.raises(mao.MaoError):  # G of another shape
        mao.dion_step(X, X.clone(), torch.zeros((64, 95), device=cuda), Q, 0.9, 1.0)
    with pytest.raises(ValueError):    # Q must be float32
        mao.dion_step(X, X.clone(), X.clone(), Q.to(torch.bfloat16), 0.9, 1.0)


@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_dion_step_out_of_place(cuda, xdt):
    """X_out receives exactly what the in-place step writes to X, X is only read, M and Q
    come out the same; X_out aliasing X is the in-place step."""
    gen = torch.Generator().manual_seed(91)
    shapes = [(256, 640), (768, 768), (300, 1000), (200, 72)]  # one rank per call: 32
    sets = [_inputs(gen, m, n, 32, "bf16", xdt, cuda) for m, n in shapes]
    X = [s[0] for s in sets]
    X0 = [x.clone() for x in X]
    M1, M2 = [s[1].clone() for s in sets], [s[1].clone() for s in sets]
    Q1, Q2 = [s[3].clone() for s in sets], [s[3].clone() for s in sets]
    G = [s[2] for s in sets]
    X_out = [torch.full_like(x, float("nan")) for x in X]
    mao.dion_step(X, M1, G, Q1, mu=0.9, lr=0.3, X_out=X_out)
    X_in = [x.clone() for x in X0]
    mao.dion_step(X_in, M2, G, Q2, mu=0.9, lr=0.3)
    X_alias = [x.clone() for x in X0]
    M3, Q3 = [s[1].clone() for s in sets], [s[3].clone() for s in sets]
    mao.dion_step(X_alias, M3, G, Q3, mu=0.9, lr=0.3, X_out=X_alias)
    mao.sync_status()
    for k in range(len(sets)):
        assert torch.equal(X[k], X0[k])
        assert torch.equal(X_out[k], X_in[k])
        assert torch.equal(X_alias[k], X_in[k])
        assert torch.equal(M1[k], M2[k]) and torch.equal(Q1[k], Q2[k])


def test_dion_rejects_bad_x_out(cuda):
    X = torch.zeros((64, 96), device=cuda)
    Q = torch.zeros((96, 8), device=cuda)
    with pytest.raises(mao.MaoError):  # X_out of another shape
        mao.dion_step(X, X.clone(), X.clone(), Q, 0.9, 1.0, X_out=torch.zeros((64, 95), device=cuda))
    with pytest.raises(mao.MaoError):  # X_out of another dtype
        mao.dion_step(X, X.clone(), X.clone(), Q, 0.9, 1.0,
                      X_out=torch.zeros((64, 96), dtype=torch.bfloat16, device=cuda))
