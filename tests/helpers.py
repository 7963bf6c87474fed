"""Shared helpers of the GPU parity tests (conversions and comparison rules)."""

import numpy as np
import torch


def to_np(t):
    """Tensor (any device, f32/bf16) -> fp32 numpy array holding the same values."""
    return t.detach().float().cpu().numpy()


def words_np(t):
    """int32 tensor of packed words -> uint32 numpy array."""
    return t.detach().cpu().numpy().view(np.uint32)


def rel_fro(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def bits_of(words, nbits):
    w = np.asarray(words, dtype="<u4")
    return np.unpackbits(w.view(np.uint8), bitorder="little")[:nbits]


def check_sign_agreement(u_gpu, u_ref, bits_gpu, strict_rms=None):
    """Signs of the GPU path vs the oracle's U.

    Every disagreement must be explained by the value error at that entry
    (|U_ref| <= |U_gpu - U_ref|), and, when `strict_rms` is given, also lie where
    |U_ref| < strict_rms * rms(U_ref). Returns the agreement fraction.
    """
    u_ref = np.asarray(u_ref, np.float64).reshape(-1)
    u_gpu = np.asarray(u_gpu, np.float64).reshape(-1)
    ref_bits = (~(u_ref < 0)).astype(np.uint8)  # oracle rule: u < 0 -> -1, else +1 (NaN: +1)
    bad = np.nonzero(bits_gpu != ref_bits)[0]
    if bad.size:
        err = np.abs(u_gpu[bad] - u_ref[bad])
        assert np.all(np.abs(u_ref[bad]) <= err + 1e-30), "sign flip not explained by the value error"
        if strict_rms is not None:
            rms = np.sqrt(np.mean(u_ref ** 2))
            assert np.all(np.abs(u_ref[bad]) < strict_rms * rms)
    return 1.0 - bad.size / u_ref.size


def rand_matrix(gen, shape, dtype, device, scale=1.0, ld=None):
    """Random matrix, optionally as a column slice of a wider buffer (row stride ld)."""
    R, C = shape
    if ld is None or ld == C:
        return (torch.randn(shape, generator=gen, device="cpu") * scale).to(dtype).to(device)
    big = (torch.randn((R, ld), generator=gen, device="cpu") * scale).to(dtype).to(device)
    return big[:, :C]


def sign_criterion(u_ref, bits_gpu, rel=1e-3):
    """The end-to-end sign criterion as stated for the step: the share of entries whose
    GPU sign equals the oracle's, and the share of the disagreements that lie where
    |U_ref| < rel * rms(U_ref). Returns (agreement, flips, share_small)."""
    u_ref = np.asarray(u_ref, np.float64).reshape(-1)
    ref_bits = (~(u_ref < 0)).astype(np.uint8)
    bad = np.nonzero(np.asarray(bits_gpu) != ref_bits)[0]
    rms = np.sqrt(np.mean(u_ref ** 2))
    small = int(np.count_nonzero(np.abs(u_ref[bad]) < rel * rms)) if bad.size else 0
    share = small / bad.size if bad.size else 1.0
    return 1.0 - bad.size / u_ref.size, int(bad.size), share
