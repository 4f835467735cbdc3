"""Pins for R(delta), the exact RoPE re-rotation of cached keys (Kamera,
gist.science/pt/paper/2606.23581, section 2, relocation bullet: an exact
algebraic operation, not a forward pass).

The pins do not retype the oracle's formula: frequencies are checked against
hand values, the pair rotation against complex multiplication, and the
operator against the closed-form identities R(d) RoPE(k, p) = RoPE(k, p + d),
R(a) R(b) = R(a + b), R(0) = I, R(-d) = R(d)^-1 and per-pair norm invariance."""
import json
import math
import os

import numpy as np
import pytest

from oracle import inv_freq, rope_absolute, relocate, round_to_bf16_bits

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")))


def test_frequencies_hand_values():
    assert np.allclose(inv_freq(2, 1e6), [1.0], rtol=0, atol=0)
    assert np.allclose(inv_freq(4, 1e4), [1.0, 0.01], rtol=1e-15)
    assert np.allclose(inv_freq(8, 16.0), [1.0, 0.5, 0.25, 0.125], rtol=1e-15)
    f = inv_freq(128, 1e6)
    assert f.shape == (64,) and f[0] == 1.0
    assert math.isclose(f[32], 1e-3, rel_tol=1e-14)          # 1e6^(-64/128)
    assert math.isclose(f[-1], 1e6 ** (-126 / 128), rel_tol=1e-14)


@pytest.mark.parametrize("case", GOLD["rotation"], ids=lambda c: c["name"])
def test_golden_rotation(case):
    y = relocate(np.array([case["x"]]), case["delta"], case["theta"])
    bits = [f"0x{b:04X}" for b in round_to_bf16_bits(y)[0]]
    assert bits == case["expect_bits"]


def test_pair_turn_is_complex_multiplication():
    rng = np.random.default_rng(1)
    d, theta = 128, 1e6
    x = rng.standard_normal((50, d))
    delta = 12345
    y = relocate(x, delta, theta)
    h = d // 2
    z = (x[:, :h] + 1j * x[:, h:]) * np.exp(1j * delta * (theta ** (-np.arange(0, d, 2) / d)))
    assert np.allclose(y[:, :h], z.real, rtol=0, atol=1e-12)
    assert np.allclose(y[:, h:], z.imag, rtol=0, atol=1e-12)


@pytest.mark.parametrize("theta,d", [(1e6, 128), (1e4, 128), (1e4, 64)])
def test_shift_identity(theta, d):
    rng = np.random.default_rng(2)
    k = rng.standard_normal((200, d))
    p = rng.integers(0, 100000, 200)
    delta = rng.integers(-65536, 65537, 200)
    lhs = np.stack([relocate(rope_absolute(k[i:i + 1], p[i:i + 1], theta), delta[i], theta)[0]
                    for i in range(200)])
    rhs = rope_absolute(k, p + delta, theta)
    err = np.linalg.norm(lhs - rhs, axis=1) / np.linalg.norm(k, axis=1)
    assert err.max() < 1e-9


def test_group_laws_and_norm():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 128))
    a, b = 31337, -65000
    assert np.array_equal(relocate(x, 0, 1e6), x)
    assert np.allclose(relocate(relocate(x, a, 1e6), b, 1e6), relocate(x, a + b, 1e6), atol=1e-10)
    assert np.allclose(relocate(relocate(x, a, 1e6), -a, 1e6), x, atol=1e-10)
    y = relocate(x, a, 1e6)
    n0 = x[:, :64] ** 2 + x[:, 64:] ** 2
    n1 = y[:, :64] ** 2 + y[:, 64:] ** 2
    assert np.allclose(n0, n1, rtol=1e-13)


def test_quarter_turn():
    # delta * theta_0 = pi/2 turns the first pair (a, b) into (-b, a)
    y = relocate(np.array([[0.75, -3.0]]), np.pi / 2, 1e4)
    assert np.allclose(y, [[3.0, 0.75]], atol=1e-15)


def test_rope_absolute_is_relocation_from_zero():
    rng = np.random.default_rng(4)
    k = rng.standard_normal((10, 64))
    p = np.arange(10) * 977
    assert np.allclose(rope_absolute(k, p, 1e4), np.stack([relocate(k[i], p[i], 1e4) for i in range(10)]),
                       atol=1e-12)
