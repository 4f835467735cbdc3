"""Pins for the M-RoPE re-rotation (multimodal RoPE of Qwen-VL-style models;
the composable-KV summary, gist.science/pt/paper/2606.17107 section 4, names
M-RoPE re-rotation for image KV).  Frequency pairs form consecutive temporal /
height / width sections; relocation turns each pair by its section's shift.

Pins: a hand-derived golden example; the shift identity
R(d) . MRoPE(k, p) = MRoPE(k, p + d) for 3-component positions, checked
against an independent complex-number formulation; equal shifts reduce to
plain RoPE; a section's shift moves only that section's pairs; group laws."""
import json
import os

import numpy as np
import pytest

from oracle import mrope_absolute, pair_shifts, relocate, rope_absolute, round_to_bf16_bits

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")))
SECTIONS = (16, 24, 24)        # Qwen2.5-VL head_dim 128


def test_golden_mrope():
    g = GOLD["mrope"]
    y = relocate(np.array([g["x"]]), tuple(g["delta"]), g["theta"], tuple(g["sections"]))
    assert [f"0x{b:04X}" for b in round_to_bf16_bits(y)[0]] == g["expect_bits"]


def test_pair_shifts_layout():
    s = pair_shifts((3, -5, 7), 64, SECTIONS)
    assert s.shape == (64,)
    assert np.all(s[:16] == 3) and np.all(s[16:40] == -5) and np.all(s[40:] == 7)
    assert np.all(pair_shifts(11, 64) == 11)
    with pytest.raises(AssertionError):
        pair_shifts((1, 2, 3), 64, (16, 24, 20))


def _mrope_complex(x, pos_thw, theta, sections):
    """Independent restatement: pair i is the complex number x_i + j x_{i+h},
    multiplied by exp(j * p_sec(i) * theta^(-2i/d))."""
    d = x.shape[-1]
    h = d // 2
    out = np.empty_like(x)
    bounds = np.cumsum((0,) + tuple(sections))
    for r in range(x.shape[0]):
        for i in range(h):
            sec = int(np.searchsorted(bounds, i, side="right") - 1)
            ang = pos_thw[r][sec] * theta ** (-2.0 * i / d)
            z = complex(x[r, i], x[r, i + h]) * complex(np.cos(ang), np.sin(ang))
            out[r, i], out[r, i + h] = z.real, z.imag
    return out


def test_absolute_mrope_matches_complex_form():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((6, 128))
    pos = rng.integers(0, 5000, (6, 3))
    assert np.allclose(mrope_absolute(x, pos, 1e6, SECTIONS), _mrope_complex(x, pos, 1e6, SECTIONS), atol=1e-10)


def test_shift_identity():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((40, 128))
    pos = rng.integers(0, 50000, (40, 3))
    for _ in range(5):
        d = tuple(int(v) for v in rng.integers(-32768, 32769, 3))
        lhs = relocate(mrope_absolute(x, pos, 1e6, SECTIONS), d, 1e6, SECTIONS)
        rhs = mrope_absolute(x, pos + np.array(d), 1e6, SECTIONS)
        assert np.max(np.abs(lhs - rhs)) < 1e-9 * np.max(np.abs(x))


def test_equal_shifts_are_plain_rope():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((10, 128))
    assert np.allclose(relocate(x, (777, 777, 777), 1e6, SECTIONS), relocate(x, 777, 1e6), atol=0)
    p = rng.integers(0, 9000, 10)
    assert np.allclose(mrope_absolute(x, np.stack([p, p, p], 1), 1e6, SECTIONS), rope_absolute(x, p, 1e6),
                       atol=1e-12)


def test_a_section_shift_moves_only_its_pairs():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((8, 128))
    a = relocate(x, (10, 20, 30), 1e6, SECTIONS)
    b = relocate(x, (10, 99, 30), 1e6, SECTIONS)
    diff = np.abs(a - b).max(axis=0)
    h = 64
    moved = np.zeros(128, bool)
    moved[16:40] = moved[16 + h:40 + h] = True
    assert np.all(diff[~moved] == 0) and np.all(diff[moved] > 0)


def test_group_laws():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((8, 128))
    d1, d2 = (100, -200, 300), (-7, 50000, 12)
    two = relocate(relocate(x, d1, 1e6, SECTIONS), d2, 1e6, SECTIONS)
    one = relocate(x, tuple(a + b for a, b in zip(d1, d2)), 1e6, SECTIONS)
    assert np.allclose(two, one, atol=1e-10)
    assert np.allclose(relocate(relocate(x, d1, 1e6, SECTIONS), tuple(-v for v in d1), 1e6, SECTIONS), x, atol=1e-10)
