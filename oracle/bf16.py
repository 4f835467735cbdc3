"""bfloat16 by definition, in fp64 (oracle; test infrastructure only).

bf16 is the upper half of an IEEE-754 binary32: 1 sign bit, 8 exponent bits,
7 stored significand bits (8 significant bits for normal numbers), subnormals
below 2^-126 with spacing 2^-133.

``round_to_bf16_bits`` rounds an fp64 value to the nearest bf16 value, ties to
the even significand, in ONE rounding step (never through fp32 first).  It is
written from that definition: find the spacing of bf16 values around |x|,
scale |x| to an integer multiple of that spacing, round to nearest-even, and
scale back.  Every step except the final ``rint`` is a multiplication by a
power of two, hence exact in fp64.
"""
from __future__ import annotations

import numpy as np

_BF16_MIN_NORMAL_EXP = -126      # smallest normal binade is [2^-126, 2^-125)
_BF16_FRAC_BITS = 7              # stored significand bits


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as fp64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_bf16_bits(x) -> np.ndarray:
    """Round fp64 values to bf16 (nearest, ties to even), returned as uint16 bits."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    neg = np.signbit(x)
    out = np.zeros(x.shape, dtype=np.uint16)

    finite = np.isfinite(x)
    nz = finite & (a > 0)
    # binade exponent E with 2^E <= a < 2^(E+1); subnormals share E = -126
    _, e = np.frexp(np.where(nz, a, 1.0))
    E = np.maximum(e.astype(np.int64) - 1, _BF16_MIN_NORMAL_EXP)
    spacing_exp = E - _BF16_FRAC_BITS
    q = np.ldexp(np.where(nz, a, 0.0), -spacing_exp)     # exact
    r = np.rint(q)                                        # nearest, ties to even
    v = np.ldexp(r, spacing_exp)                          # exact
    overflow = nz & (v >= 2.0 ** 128)
    v32 = np.where(overflow | ~nz, 0.0, v).astype(np.float32)   # exactly representable
    mag = (v32.view(np.uint32) >> 16).astype(np.uint16)
    mag = np.where(overflow, np.uint16(0x7F80), mag)
    mag = np.where(np.isinf(x), np.uint16(0x7F80), mag)
    out = np.where(neg, mag | np.uint16(0x8000), mag).astype(np.uint16)
    out = np.where(np.isnan(x), np.uint16(0x7FC0), out).astype(np.uint16)
    return out


def bf16_ord(bits) -> np.ndarray:
    """Map bf16 bit patterns to integers that are monotone in value, with +0 and
    -0 both mapped to 0, so that adjacent finite bf16 values differ by 1."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_distance(a_bits, b_bits) -> np.ndarray:
    """Number of bf16 steps between two bf16 bit patterns (finite values)."""
    return np.abs(bf16_ord(a_bits) - bf16_ord(b_bits))


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bf16 values in the binade of |x| (2^-133 below the normal range)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    E = np.maximum(e.astype(np.int64) - 1, _BF16_MIN_NORMAL_EXP)
    E = np.where(a > 0, E, _BF16_MIN_NORMAL_EXP)
    return np.ldexp(1.0, E - _BF16_FRAC_BITS)
