"""fp64 oracle of the Muon / Sign-Muon step (test infrastructure, see package doc).

Stages, in the order [SignMuon] §2 "Fluxo Algorítmico (Distribuído)" gives them:

  1. local momentum of each worker, then its polar factor by Newton–Schulz;
  2. entrywise sign of the polar factor, values in {-1, +1};
  3. the 1-bit all-gather variant: signs packed one bit per entry;
  4. majority vote sign(sum_m S^(m)) and the update W <- W - eta * S_bar.

Readings taken where the sources are silent (each is listed with its reason in
the design notes of the repository):

* momentum is the heavy-ball form M <- mu*M + G, as written in [Dion] §"Ablation"
  (the baseline without error feedback); it is one fp32 fused multiply-add,
  then a round to the storage type;
* the polar factor is approximated by the odd-polynomial Newton–Schulz iteration
  X <- a X + (b A + c A^2) X with A = X X^T, three matrix products per iteration
  as [Megatron] §"分散ニュートン・シュルツ" counts them, on the Frobenius-normalised
  momentum ([SignMuon] §4 "nanoGPT" names Frobenius scaling), eps = 1e-7;
* the iteration runs on the orientation with rows <= columns (a tall matrix is
  transposed first and the result transposed back);
* sign(u) is -1 for u < 0 and +1 otherwise (+0, -0 and NaN give +1);
* bits are packed row-major in the matrix's own orientation, least significant
  bit first, 32 entries per uint32 word, ceil(N/32) words, padding bits 0;
  bit = 1 encodes +1;
* a tied vote (even number of workers) gives +1;
* the update is one fp32 fused multiply-add W + (-eta) * D, then a round to the
  storage type (D = +-1 for Sign-Muon, D = U for Muon).
"""

import numpy as np

from .rounding import bf16_rne, fma_f32

# Quintic coefficients (a, b, c), the same at every iteration. The sources print
# no coefficients; these are the widely used Muon quintic.
QUINTIC = (3.4445, -4.7750, 2.0315)
# Cubic Newton–Schulz, p(s) = 1.5 s - 0.5 s^3: converges to the polar factor.
CUBIC = (1.5, -0.5, 0.0)


def _store(x32, dtype):
    if dtype == "f32":
        return np.asarray(x32, dtype=np.float32)
    if dtype == "bf16":
        return bf16_rne(x32)
    raise ValueError(dtype)


def momentum(M, G, mu, store="f32"):
    """Local momentum M <- mu*M + G of one worker ([SignMuon] §2 step 1, form from [Dion]).

    One fp32 fused multiply-add per element, then a round to ``store``.
    M and G are fp32 arrays holding values of their storage types.
    """
    r = fma_f32(np.float32(mu), np.asarray(M, np.float32), np.asarray(G, np.float32))
    return _store(r, store)


def frobenius_normalise(X, eps=1e-7):
    """X / (||X||_F + eps) in fp64 ([SignMuon] §4 names Frobenius scaling)."""
    X = np.asarray(X, dtype=np.float64)
    return X / (np.sqrt(np.sum(X * X)) + eps)


def _coeff_list(coeffs, steps):
    coeffs = list(coeffs)
    if len(coeffs) == 3 and not isinstance(coeffs[0], (tuple, list, np.ndarray)):
        return [tuple(coeffs)] * steps
    if len(coeffs) != steps:
        raise ValueError("need one (a, b, c) triple per step")
    return [tuple(t) for t in coeffs]


def newton_schulz(M, steps=5, coeffs=QUINTIC, eps=1e-7):
    """Polar direction of M by Newton–Schulz ([SignMuon] §2 "Mecanismo Central" 1).

    fp64 throughout. Per iteration the three matrix products of
    [Megatron] §"分散ニュートン・シュルツ": A = X X^T, then B = b A + c (A A),
    then X <- a X + B X.
    """
    X = np.asarray(M, dtype=np.float64)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    X = frobenius_normalise(X, eps)
    for a, b, c in _coeff_list(coeffs, steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if tall else X


def blockwise_newton_schulz(M, block_rows, block_cols, steps=5, coeffs=QUINTIC, eps=1e-7):
    """Blockwise orthogonalisation ([Megatron] §"分散モード", blockwise paragraph): each
    block of a block_rows x block_cols grid (the last block row / column ragged) is what one
    rank owns, and is orthogonalised on its own (its own Frobenius norm, its own
    Newton–Schulz). This is not the orthogonalisation of the whole matrix."""
    M = np.asarray(M, dtype=np.float64)
    R, C = M.shape
    out = np.empty_like(M)
    for i0 in range(0, R, block_rows):
        for j0 in range(0, C, block_cols):
            blk = M[i0:i0 + block_rows, j0:j0 + block_cols]
            out[i0:i0 + block_rows, j0:j0 + block_cols] = newton_schulz(blk, steps, coeffs, eps)
    return out


def sign_of(U):
    """Entrywise sign in {-1, +1} ([SignMuon] §2 step 2); u < 0 -> -1, else +1."""
    U = np.asarray(U)
    return np.where(U < 0, -1, 1).astype(np.int8)


def pack_signs_loop(S):
    """One bit per entry ([SignMuon] §2 step 3), plain Python loop (small inputs).

    Row-major order, bit k of the flattened matrix goes to word k // 32, bit
    k % 32 (least significant first); bit = 1 encodes +1.
    """
    flat = [int(v) for v in np.asarray(S).reshape(-1)]
    nwords = (len(flat) + 31) // 32
    words = [0] * nwords
    for k, v in enumerate(flat):
        if v > 0:
            words[k // 32] |= 1 << (k % 32)
    return np.array(words, dtype=np.uint32)


def pack_signs(S):
    """Vectorised form of ``pack_signs_loop`` (numpy packbits, little bit order)."""
    bits = (np.asarray(S).reshape(-1) > 0).astype(np.uint8)
    nwords = (bits.size + 31) // 32
    padded = np.zeros(nwords * 32, dtype=np.uint8)
    padded[: bits.size] = bits
    by = np.packbits(padded, bitorder="little")
    return by.view("<u4").astype(np.uint32)


def unpack_signs(words, nbits):
    """Inverse of ``pack_signs``: words -> int8 array of nbits signs in {-1, +1}."""
    w = np.asarray(words, dtype="<u4")
    bits = np.unpackbits(w.view(np.uint8), bitorder="little")[:nbits]
    return np.where(bits == 1, 1, -1).astype(np.int8)


def majority_vote(worker_words, nbits):
    """Majority vote sign(sum_m S^(m)) over packed worker buffers ([SignMuon] §2 step 4).

    ``worker_words`` is [W_n][nwords] (the all-gather result layout). Signs are
    unpacked to +-1, summed as integers, and the sum's sign taken with ties -> +1.
    Returns the packed vote.
    """
    ww = np.asarray(worker_words, dtype=np.uint32)
    total = np.zeros(nbits, dtype=np.int64)
    for m in range(ww.shape[0]):
        total += unpack_signs(ww[m], nbits).astype(np.int64)
    vote = np.where(total >= 0, 1, -1).astype(np.int8)
    return pack_signs(vote)


def int8_sum_vote(S_workers):
    """All-reduce variant of the vote ([SignMuon] §2 step 3 "Variante All-Reduce"):
    signs travel as int8 +-1, an integer SUM over the workers gives sum_m S^(m), and the
    local threshold sign(.) with ties -> +1 gives S_bar. Returns (sums, S_bar)."""
    total = np.zeros(np.asarray(S_workers[0]).shape, dtype=np.int64)
    for S in S_workers:
        total += np.asarray(S, dtype=np.int64)
    return total, np.where(total >= 0, 1, -1).astype(np.int8)


def post_vote_polar(S_bar, steps=5, coeffs=QUINTIC, eps=1e-7):
    """Optional local polar step on the aggregated sign matrix ([SignMuon] §2 step 5):
    Newton-Schulz applied to S_bar (+-1 entries) before the update."""
    return newton_schulz(np.asarray(S_bar, dtype=np.float64), steps, coeffs, eps)


def apply_update(W, D, lr, store="f32"):
    """W <- W - eta * D as one fp32 fused multiply-add, rounded to ``store``.

    [SignMuon] §2 step 4 (D = S_bar in {-1, +1}); the Muon step uses D = U as stored.
    """
    r = fma_f32(-np.float32(lr), np.asarray(D, np.float32), np.asarray(W, np.float32))
    return _store(r, store)


def apply_update_f64(W, D, lr):
    """W - eta * D in fp64 (for end-to-end comparisons with an fp64 direction)."""
    return np.asarray(W, np.float64) - float(np.float32(lr)) * np.asarray(D, np.float64)


def sign_muon_step(W, Ms, Gs, mu, lr, steps=5, coeffs=QUINTIC, eps=1e-7,
                   m_store="f32", w_store="f32", variant="bits", post_polar=False):
    """One Sign-Muon step over W_n simulated workers ([SignMuon] §2).

    variant "bits": the 1-bit all-gather variant (packed words, vote on the words);
    variant "int8": the integer SUM all-reduce variant (int8 sums, then the threshold).
    post_polar: the optional local polar step of [SignMuon] §2 step 5; the update is then
    W - eta * polar(S_bar) in fp64 (Newton–Schulz with the same steps and coefficients).

    Returns a dict with every intermediate: per-worker momentum, polar factor U, signs,
    the aggregation's buffers, S_bar, (U_bar) and the updated W.
    """
    if variant not in ("bits", "int8"):
        raise ValueError(variant)
    Wn = len(Ms)
    nbits = int(np.asarray(W).size)
    M_new = [momentum(Ms[m], Gs[m], mu, m_store) for m in range(Wn)]
    U = [newton_schulz(M_new[m], steps, coeffs, eps) for m in range(Wn)]
    S = [sign_of(u) for u in U]
    out = {"M": M_new, "U": U, "S": S}
    if variant == "bits":
        words = np.stack([pack_signs(s) for s in S])
        vote = majority_vote(words, nbits)
        S_bar = unpack_signs(vote, nbits).reshape(np.asarray(W).shape)
        out.update(words=words, vote=vote)
    else:
        sums, S_bar = int8_sum_vote(S)
        out.update(sums=sums)
    out["S_bar"] = S_bar
    if post_polar:
        out["U_bar"] = post_vote_polar(S_bar, steps, coeffs, eps)
        out["W"] = apply_update_f64(W, out["U_bar"], lr)
    else:
        out["W"] = apply_update(W, S_bar, lr, w_store)
    return out


def muon_step(Ws, Ms, Gs, mu, lr, steps=5, coeffs=QUINTIC, eps=1e-7,
              m_store="f32"):
    """One Muon step over a batch of matrices: momentum, polar factor, W - eta*U (fp64)."""
    M_new = [momentum(M, G, mu, m_store) for M, G in zip(Ms, Gs)]
    U = [newton_schulz(M, steps, coeffs, eps) for M in M_new]
    W_new = [apply_update_f64(W, u, lr) for W, u in zip(Ws, U)]
    return {"M": M_new, "U": U, "W": W_new}


def ns_dense_flops(rows, cols, steps):
    """Dense-count flops of Newton–Schulz: (4 m^2 n + 2 m^3) per iteration, m <= n."""
    m, n = min(rows, cols), max(rows, cols)
    return steps * (4 * m * m * n + 2 * m ** 3)
