"""Pins for the patch-formation side of the oracle (Kamera,
gist.science/pt/paper/2606.23581, section 2, patch bullet): the deficit
Delta = KV(B|A) - R(delta) KV(B|empty) and its truncated SVD.

The deficit is checked against absolute-position RoPE (a cache encoded at
positions p + delta has zero deficit against the same cache encoded at p), so
a wrong sign, pairing or frame in the relocation shows up; a planted low-rank
conditioning term with known singular values pins the SVD and the
Eckart-Young tail by closed form."""
import numpy as np
import pytest

from oracle import (conditioning_deficit, eckart_young_tail, inv_freq, rope_absolute, row_layout, svd_patch)


def _keys(rng, T, H, d, pos, theta, raw=None):
    raw = rng.standard_normal((T, H * d)) if raw is None else raw
    out = np.concatenate([rope_absolute(raw[:, h * d:(h + 1) * d], pos, theta) for h in range(H)], axis=1)
    return raw, out


@pytest.mark.parametrize("delta", [1, 517, -300, 40000])
def test_deficit_vanishes_for_a_pure_shift(delta):
    rng = np.random.default_rng(41)
    T, H, d, theta = 23, 2, 64, 1e4
    pos = np.arange(T) + 1000
    raw, canon = _keys(rng, T, H, d, pos, theta)
    _, cond = _keys(rng, T, H, d, pos + delta, theta, raw)
    dk = conditioning_deficit(cond, canon, delta, theta, row_layout("gqa", "k", n_heads=H, head_dim=d))
    assert np.max(np.abs(dk)) < 1e-9
    # the same pair with the shift's sign flipped is far from zero
    wrong = conditioning_deficit(cond, canon, -delta, theta, row_layout("gqa", "k", n_heads=H, head_dim=d))
    assert np.max(np.abs(wrong)) > 0.1


def test_deficit_of_values_and_of_the_mla_latent_is_a_plain_difference():
    rng = np.random.default_rng(42)
    T = 19
    a, b = rng.standard_normal((T, 96)), rng.standard_normal((T, 96))
    dv = conditioning_deficit(a, b, 77, 1e4, row_layout("gqa", "v", n_heads=3, head_dim=32))
    assert np.array_equal(dv, a - b)
    # MLA row: c_KV (first 32) differs plainly; k_rope (last 64) is relocated first
    lora, rope, theta, delta = 32, 64, 1e4, 250
    pos = np.arange(T)
    raw_r = rng.standard_normal((T, rope))
    canon = np.concatenate([rng.standard_normal((T, lora)), rope_absolute(raw_r, pos, theta)], axis=1)
    cond = np.concatenate([canon[:, :lora] + 0.5, rope_absolute(raw_r, pos + delta, theta)], axis=1)
    dm = conditioning_deficit(cond, canon, delta, theta, row_layout("mla", "k", kv_lora_dim=lora, rope_dim=rope))
    assert np.allclose(dm[:, :lora], 0.5, atol=1e-12, rtol=0)
    assert np.max(np.abs(dm[:, lora:])) < 1e-9


def test_planted_low_rank_conditioning_is_recovered():
    """cond = R(delta) canon + P with P = sum_i s_i a_i b_i^T (orthonormal a, b):
    the deficit is P, the rank-r SVD patch rebuilds it, and truncating to m < r
    leaves exactly sum_{i >= m} s_i^2 (Eckart-Young, closed form)."""
    rng = np.random.default_rng(43)
    T, H, d, theta, delta, r = 64, 2, 32, 1e6, -1234, 6
    pos = np.arange(T)
    raw, canon = _keys(rng, T, H, d, pos, theta)
    _, shifted = _keys(rng, T, H, d, pos + delta, theta, raw)
    a = np.linalg.qr(rng.standard_normal((T, r)))[0]
    b = np.linalg.qr(rng.standard_normal((H * d, r)))[0]
    s = np.array([9.0, 5.0, 3.0, 2.0, 1.0, 0.5])
    planted = (a * s) @ b.T
    dk = conditioning_deficit(shifted + planted, canon, delta, theta, row_layout("gqa", "k", n_heads=H, head_dim=d))
    assert np.allclose(dk, planted, atol=1e-9, rtol=0)
    u, w = svd_patch(dk, r)
    assert np.allclose(u @ w.T, planted, atol=1e-8, rtol=0)
    for m in range(r + 1):
        u, w = svd_patch(dk, m)
        assert abs(np.sum((dk - u @ w.T) ** 2) - np.sum(s[m:] ** 2)) < 1e-8
        assert abs(eckart_young_tail(dk, m) - np.sum(s[m:] ** 2)) < 1e-8
    # the factors: W has orthonormal columns (the right singular vectors), U carries the singular values
    u, w = svd_patch(dk, 4)
    assert np.allclose(w.T @ w, np.eye(4), atol=1e-12)
    assert np.allclose(np.linalg.norm(u, axis=0), s[:4], rtol=1e-10)


def test_inverse_frequencies_used_by_the_deficit():
    # one pair per head (d = 2): the whole row turns by delta * theta^0 = delta radians
    x = np.array([[1.0, 0.0]])
    d1 = conditioning_deficit(np.array([[np.cos(3.0), np.sin(3.0)]]), x, 3, 1e4, row_layout("gqa", "k", n_heads=1, head_dim=2))
    assert np.max(np.abs(d1)) < 1e-15
    assert inv_freq(2, 1e4)[0] == 1.0


# --------------------------------------------------------------------------- #
# Orbit patch: the deficit averaged over orderings
# --------------------------------------------------------------------------- #

def test_orbit_deficit_hand_example():
    """d = 2, theta_0 = 1, two orderings with shifts +1 and -1, x = (1, 0).
    The conditioned caches are the shifted x plus (0.5, 0) and (0.25, 0.5):
    the mean deficit is (0.375, 0.25).  With zero conditioned caches the
    deficit is -Rbar x where Rbar averages the two rotations: mean cos = cos 1,
    mean sin = 0, so -Rbar x = (-cos 1, 0) = (-0.5403023058681398, 0)."""
    from oracle import orbit_deficit
    lay = row_layout("gqa", "k", n_heads=1, head_dim=2)
    x = np.array([[1.0, 0.0]])
    c1, s1 = 0.5403023058681398, 0.8414709848078965
    conds = [np.array([[c1 + 0.5, s1]]), np.array([[c1 + 0.25, -s1 + 0.5]])]
    d = orbit_deficit(conds, x, [1, -1], 1e4, lay)
    assert np.allclose(d, [[0.375, 0.25]], atol=1e-15, rtol=0)
    z = orbit_deficit([np.zeros((1, 2)), np.zeros((1, 2))], x, [1, -1], 1e4, lay)
    assert np.allclose(z, [[-c1, 0.0]], atol=1e-15, rtol=0)


def test_orbit_of_pure_shifts_is_zero_and_planted_terms_average():
    from oracle import orbit_deficit
    rng = np.random.default_rng(44)
    T, H, d, theta = 40, 2, 64, 1e6
    pos = np.arange(T) + 77
    deltas = [0, 1500, -700, 4096]
    raw, canon = _keys(rng, T, H, d, pos, theta)
    lay = row_layout("gqa", "k", n_heads=H, head_dim=d)
    shifted = [_keys(rng, T, H, d, pos + dl, theta, raw)[1] for dl in deltas]
    assert np.max(np.abs(orbit_deficit(shifted, canon, deltas, theta, lay))) < 1e-9
    planted = [rng.standard_normal((T, H * d)) for _ in deltas]
    got = orbit_deficit([s + p for s, p in zip(shifted, planted)], canon, deltas, theta, lay)
    assert np.allclose(got, sum(planted) / len(planted), atol=1e-9, rtol=0)
    # a single ordering is the plain deficit
    one = orbit_deficit([shifted[1] + planted[1]], canon, [deltas[1]], theta, lay)
    assert np.allclose(one, planted[1], atol=1e-9, rtol=0)
    with pytest.raises(ValueError):
        orbit_deficit([canon], canon, [1, 2], theta, lay)
