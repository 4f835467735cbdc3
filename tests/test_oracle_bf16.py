"""Pins for the oracle's bf16 arithmetic: exhaustive round trips, every
midpoint of the bf16 grid, agreement with torch's float32 -> bf16 conversion
(an independent library routine), single (not double) rounding, overflow,
subnormals, and the ulp metric."""
import numpy as np
import pytest
import torch

from oracle import bf16_bits_to_f64, round_to_bf16_bits, bf16_ord, ulp_distance, bf16_ulp

ALL = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
FINITE = ALL[((ALL.astype(np.uint32) >> 7) & 0xFF) != 0xFF]


def test_decode_matches_float32_upper_half():
    v = bf16_bits_to_f64(np.array([0x3F80, 0xBF80, 0x4040, 0x0001, 0x7F7F], np.uint16))
    assert v[0] == 1.0 and v[1] == -1.0 and v[2] == 3.0
    assert v[3] == 2.0 ** -133
    assert v[4] == (2 - 2 ** -7) * 2.0 ** 127


def test_round_trip_every_finite_pattern():
    back = round_to_bf16_bits(bf16_bits_to_f64(FINITE))
    assert np.array_equal(back, FINITE)  # includes +0 / -0 and all subnormals


def test_every_positive_midpoint_ties_to_even_and_breaks_correctly():
    lo = FINITE[(FINITE < 0x7F7F)]
    lo = lo[lo < 0x8000]
    hi = (lo.astype(np.uint32) + 1).astype(np.uint16)
    a, b = bf16_bits_to_f64(lo), bf16_bits_to_f64(hi)
    mid = (a + b) / 2  # exact in fp64
    even = np.where(lo & 1, hi, lo)
    assert np.array_equal(round_to_bf16_bits(mid), even)
    assert np.array_equal(round_to_bf16_bits(np.nextafter(mid, np.inf)), hi)
    assert np.array_equal(round_to_bf16_bits(np.nextafter(mid, -np.inf)), lo)
    # negative side mirrors the positive side
    assert np.array_equal(round_to_bf16_bits(-mid), even | np.uint16(0x8000))


def test_agrees_with_torch_float32_conversion():
    rng = np.random.default_rng(5)
    f = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(50000) * 1e-39).astype(np.float32),   # fp32 subnormals
        (rng.standard_normal(50000) * 1e37).astype(np.float32),
        rng.integers(0, 2 ** 32, 100000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    f = f[np.isfinite(f)]
    ours = round_to_bf16_bits(f.astype(np.float64))
    theirs = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_single_rounding_not_through_float32():
    # 1 + 2^-8 is the midpoint between bf16 1.0 (even) and 1 + 2^-7.  A value a
    # hair above it must round up; rounding to fp32 first would land on the
    # midpoint and then tie down to 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert np.float32(x) == np.float32(1.0 + 2.0 ** -8)
    assert round_to_bf16_bits(x) == 0x3F81


def test_overflow_and_specials():
    top = (2 - 2 ** -7) * 2.0 ** 127
    assert round_to_bf16_bits(top) == 0x7F7F
    assert round_to_bf16_bits((2 - 2 ** -8) * 2.0 ** 127) == 0x7F80   # midpoint to inf ties away
    assert round_to_bf16_bits(np.nextafter((2 - 2 ** -8) * 2.0 ** 127, 0)) == 0x7F7F
    assert round_to_bf16_bits(-1e300) == 0xFF80
    assert round_to_bf16_bits(np.inf) == 0x7F80
    assert round_to_bf16_bits(-0.0) == 0x8000
    assert round_to_bf16_bits(2.0 ** -134) == 0x0000      # half the smallest subnormal: tie to even 0
    assert round_to_bf16_bits(3 * 2.0 ** -134) == 0x0002  # 1.5 spacings -> 2 (even)


def test_ulp_metric():
    assert ulp_distance(np.uint16(0x3F80), np.uint16(0x3F81)) == 1
    assert ulp_distance(np.uint16(0x0000), np.uint16(0x8000)) == 0
    assert ulp_distance(np.uint16(0x0001), np.uint16(0x8001)) == 2
    assert ulp_distance(np.uint16(0x3F7F), np.uint16(0x3F80)) == 1   # across a binade
    o = bf16_ord(FINITE)
    v = bf16_bits_to_f64(FINITE)
    order = np.argsort(v, kind="stable")
    assert np.all(np.diff(o[order]) >= 0)
    assert bf16_ulp(1.0) == 2.0 ** -7 and bf16_ulp(1.99) == 2.0 ** -7 and bf16_ulp(2.0) == 2.0 ** -6
    assert bf16_ulp(1e-45) == 2.0 ** -133
