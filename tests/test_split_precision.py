"""The accuracy of the bf16 part products behind Dion's Cholesky QR, in exact arithmetic.

A value x (fp32) is split into bf16 parts x = hi + mid + lo with hi = bf16(x),
mid = bf16(x - hi), lo = bf16(x - hi - mid) (round to nearest even; each difference is
exact in fp32). The Gram matrix keeps six part products and the multiply by W = L^-1 three:
  S ~ hh + hm + mh + hl + lh + mm               (error below 2^-26 of |P|^2)
  P W^T ~ P_hi W_hi^T + P_hi W_lo^T + P_mid W_hi^T   (about 2^-17 relative)
Here the part products are summed in fp64, so only the splitting is measured; the GPU adds
fp32 accumulation on top. The bf16 rounding is emulated on the fp32 bit patterns.
"""

import numpy as np
import pytest


def bf16(x):
    """Round fp32 values to the nearest bf16 (ties to even), returned as fp32."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def parts(x):
    x = np.asarray(x, dtype=np.float32)
    hi = bf16(x)
    d = (x - hi).astype(np.float32)  # exact
    mid = bf16(d)
    lo = bf16((d - mid).astype(np.float32))
    return hi, mid, lo


def test_bf16_emulation_is_round_to_nearest_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even significand (1)
    assert bf16(np.float32(1 + 2.0 ** -8)) == 1.0
    assert bf16(np.float32(1 + 3 * 2.0 ** -8)) == np.float32(1 + 2.0 ** -6)
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    assert np.all(np.abs(bf16(x) - x) <= 2.0 ** -8 * np.abs(x))


@pytest.mark.parametrize("scale", [1.0, 1e-3, 1e3])
def test_three_parts_carry_fp32_values(scale):
    x = (np.random.default_rng(1).standard_normal(20000) * scale).astype(np.float32)
    hi, mid, lo = parts(x)
    rest = x.astype(np.float64) - hi - mid - lo
    assert np.all(np.abs(rest) <= 2.0 ** -24 * np.abs(x.astype(np.float64)))


@pytest.mark.parametrize("m,r,decay", [(300, 48, 0.0), (768, 64, 3.0), (1000, 32, 6.0)])
def test_gram_from_six_part_products(m, r, decay):
    rng = np.random.default_rng(m + r)
    # columns with a spread of norms (condition up to about 10^decay)
    P = (rng.standard_normal((m, r)) * np.logspace(0, -decay, r)).astype(np.float32)
    hi, mid, lo = (p.astype(np.float64) for p in parts(P))
    S = P.astype(np.float64).T @ P.astype(np.float64)
    hh, hm, hl, mm = hi.T @ hi, hi.T @ mid, hi.T @ lo, mid.T @ mid
    S6 = hh + hm + hm.T + hl + hl.T + mm
    # entrywise against the scale of the entry's row and column (Cauchy-Schwarz bound)
    norms = np.sqrt(np.diag(S))
    err = np.abs(S6 - S) / np.outer(norms, norms)
    assert err.max() <= 2.0 ** -26  # measured about 2^-29; leaving out mm or hl gives 2^-18
    # the three dropped products are what is left
    left = S - S6
    dropped = mid.T @ lo + lo.T @ mid + lo.T @ lo
    assert np.abs(left - dropped).max() <= 2.0 ** -26 * np.abs(S).max()


def test_multiply_from_three_part_products():
    rng = np.random.default_rng(7)
    m, r = 500, 64
    P = rng.standard_normal((m, r)).astype(np.float32)
    L = np.linalg.cholesky(P.astype(np.float64).T @ P.astype(np.float64))
    W = np.linalg.inv(L).astype(np.float32)
    Ph, Pm, _ = (p.astype(np.float64) for p in parts(P))
    Wh, Wl, _ = (w.astype(np.float64) for w in parts(W))
    got = Ph @ Wh.T + Ph @ Wl.T + Pm @ Wh.T
    want = P.astype(np.float64) @ W.astype(np.float64).T
    assert np.linalg.norm(got - want) <= 2.0 ** -16 * np.linalg.norm(want)  # measured 2^-17.8
    # and the result is orthonormal to that accuracy
    assert np.abs(got.T @ got - np.eye(r)).max() <= 1e-3
