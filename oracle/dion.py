"""fp64 oracle of one Dion step (test infrastructure, see the package doc).

Source: [Dion] "대규모 AI 모델 학습을 10배 빠르게: Dion 옵티마이저를 사용한 분산 학습"
(dsdanielpark.github.io), section on the algorithm (buffer, single power iteration,
error-feedback momentum, column normalisation, orthonormal update).

The step, for a parameter matrix X (m x n), momentum M, gradient G and the previous
right factor Q_prev (n x r):

  B     = M + G                                 temporary buffer
  P     = orthonormalise(B Q_prev)              single power iteration, warm-started
  R     = B^T P                                 (m x r and n x r)
  M_new = B - (1 - mu) P R^T                    error feedback
  Q     = ColumnNormalize(R)
  X_new = X - lr P Q^T

Readings where the page is silent (listed with their reasons in the design notes):
* the power iteration is P = B Q_prev, then an orthonormal basis of P's columns, then
  R = B^T P (so that P R^T is the projection P P^T B of B onto span(P));
* that basis is the Q factor of the thin QR decomposition with a positive diagonal in
  the triangular factor (Gram–Schmidt order of the columns);
* ColumnNormalize divides each column by its Euclidean norm; a zero column stays zero;
* the update has no extra shape factor (X - lr P Q^T as printed).
"""

import numpy as np


def orthonormalise_columns(P):
    """Thin QR of P (m x r, m >= r), returning the Q factor with diag(R) > 0."""
    P = np.asarray(P, dtype=np.float64)
    Qf, Rf = np.linalg.qr(P, mode="reduced")
    s = np.where(np.diag(Rf) < 0, -1.0, 1.0)
    return Qf * s


def column_normalize(R):
    """Each column divided by its Euclidean norm (zero columns stay zero)."""
    R = np.asarray(R, dtype=np.float64)
    c = np.sqrt(np.sum(R * R, axis=0))
    return np.divide(R, c, out=np.zeros_like(R), where=c > 0)


def dion_step(X, M, G, Q_prev, mu, lr):
    """One Dion step in fp64. Returns every intermediate (B, P, R, M, Q, X)."""
    X = np.asarray(X, dtype=np.float64)
    B = np.asarray(M, dtype=np.float64) + np.asarray(G, dtype=np.float64)
    P = orthonormalise_columns(B @ np.asarray(Q_prev, dtype=np.float64))
    R = B.T @ P
    M_new = B - (1.0 - mu) * (P @ R.T)
    Q = column_normalize(R)
    X_new = X - lr * (P @ Q.T)
    return {"B": B, "P": P, "R": R, "M": M_new, "Q": Q, "X": X_new}
