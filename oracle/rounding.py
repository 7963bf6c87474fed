"""Exact rounding rules used by the oracle (test infrastructure, see package doc).

The optimizer step stores tensors in fp32 or bfloat16 and does its per-element
arithmetic in fp32. The oracle reproduces that arithmetic exactly so that the
stages whose result is unique (momentum, update) can be compared bit for bit:

* ``to_f32``   IEEE round-to-nearest-even from fp64 to fp32 (numpy's cast).
* ``bf16_rne`` round-to-nearest-even from fp32 to bfloat16 (8 significant bits),
               written out on the bit pattern.
* ``fma_f32``  a fused multiply-add in fp32: the exact value a*b + c rounded once.
"""

from fractions import Fraction

import numpy as np


def to_f32(x):
    """Round fp64 (or any real array) to fp32, nearest-even (IEEE conversion)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def bf16_rne(x):
    """Round fp32 values to bfloat16, nearest-even; returns fp32 holding bf16 values.

    bfloat16 keeps the upper 16 bits of the fp32 pattern. Round-to-nearest-even
    adds 0x7FFF plus the lowest kept bit to the pattern and truncates. Overflow
    goes to infinity; NaN stays NaN (quiet, sign kept).
    """
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep_lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    nan = np.isnan(a)
    if nan.any():
        quiet = (u.astype(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x00400000)
        r = np.where(nan, quiet, r)
    return r.view(np.float32).reshape(a.shape)


def _f32_neighbour_toward(r, s):
    """The fp32 number adjacent to r on the side of s (r itself where s == r)."""
    up = np.nextafter(r, np.float32(np.inf))
    down = np.nextafter(r, np.float32(-np.inf))
    r64 = r.astype(np.float64)
    return np.where(s > r64, up, np.where(s < r64, down, r))


def fma_f32(a, b, c):
    """fp32 fused multiply-add: round-to-nearest-even of the exact a*b + c.

    a*b of two fp32 numbers is exact in fp64 (24 + 24 significant bits <= 53).
    The fp64 sum s = fl64(a*b + c) is then rounded once more to fp32. That second
    rounding can differ from rounding the exact value only when s lands exactly on
    the midpoint between two adjacent fp32 numbers (fp64 rounding is monotone, so
    otherwise s and the exact value lie on the same side of every midpoint). For
    those elements the exact value is recomputed with rational arithmetic and
    rounded by comparing it with the midpoint.
    """
    a32 = np.asarray(a, dtype=np.float32)
    b32 = np.asarray(b, dtype=np.float32)
    c32 = np.asarray(c, dtype=np.float32)
    a32, b32, c32 = np.broadcast_arrays(a32, b32, c32)
    shape = a32.shape
    a32, b32, c32 = (np.atleast_1d(t).reshape(-1) for t in (a32, b32, c32))
    p = a32.astype(np.float64) * b32.astype(np.float64)
    s = p + c32.astype(np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        r = s.astype(np.float32)
        nb = _f32_neighbour_toward(r, s)
        mid = (r.astype(np.float64) + nb.astype(np.float64)) / 2.0
    suspect = np.isfinite(r) & np.isfinite(nb) & (s != r.astype(np.float64)) & (s == mid)
    if suspect.any():
        r = np.array(r, copy=True)
        for idx in zip(*np.nonzero(suspect)):
            exact = Fraction(float(a32[idx])) * Fraction(float(b32[idx])) + Fraction(float(c32[idx]))
            lo, hi = r[idx], nb[idx]
            m = Fraction(float(mid[idx]))
            if exact == m:
                # tie: the candidate with an even last significand bit
                lo_even = (np.array(lo, np.float32).view(np.uint32) & 1) == 0
                r[idx] = lo if lo_even else hi
            elif (exact > m) == (Fraction(float(hi)) > m):
                r[idx] = hi
            else:
                r[idx] = lo
    return r.reshape(shape)
