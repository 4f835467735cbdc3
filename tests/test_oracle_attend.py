"""Pins for the decode-attention oracle over relocated, patched chunks (the
fused read-side use of the Kamera operator, gist.science/pt/paper/2606.23581,
section 2): absolute-position RoPE (a relocated chunk attends exactly like one
encoded at its new positions), closed forms (one token; equal keys give the
mean of the values; a patch that only moves one value row), the grouped-query
head mapping, and a brute-force softmax written out with scalar loops."""
import math

import numpy as np
import pytest

from oracle import attend_relocated, attention, relocated_chunk, rope_absolute, round_to_bf16_bits, bf16_bits_to_f64


def _bits(x):
    return round_to_bf16_bits(np.asarray(x, dtype=np.float64))


def test_relocated_chunk_attends_like_keys_encoded_at_the_new_positions():
    """Keys cached at positions p and relocated by delta are the keys encoded
    at p + delta: R(delta) x = RoPE(x, delta) per head, and the attention over
    the relocated chunk matches the attention over keys encoded at p + delta
    (up to the bf16 rounding of the cached keys)."""
    rng = np.random.default_rng(61)
    T, H, Hq, d, theta, delta = 37, 2, 6, 64, 1e4, 1234
    pos = np.arange(T) + 100
    raw = rng.standard_normal((T, H, d))
    canon_bits = _bits(np.concatenate([rope_absolute(raw[:, h], pos, theta) for h in range(H)], axis=1))
    v = rng.standard_normal((T, H * d))
    q = rng.standard_normal(Hq * d)
    k_hat, v_hat = relocated_chunk(canon_bits, _bits(v), delta, theta, H, d)
    canon = bf16_bits_to_f64(canon_bits)
    by_rope = np.concatenate([rope_absolute(canon[:, h * d:(h + 1) * d], np.full(T, delta), theta)
                              for h in range(H)], axis=1)
    assert np.allclose(k_hat, by_rope, atol=1e-9, rtol=0)
    assert np.array_equal(v_hat, bf16_bits_to_f64(_bits(v)))          # values do not turn
    moved = np.concatenate([rope_absolute(raw[:, h], pos + delta, theta) for h in range(H)], axis=1)
    got = attention(q, k_hat, v_hat, Hq, H, d, 0.125)
    want = attention(q, moved, v_hat, Hq, H, d, 0.125)
    assert np.max(np.abs(got - want)) < 0.05


def test_one_token_context_returns_its_value():
    rng = np.random.default_rng(62)
    H, Hq, d = 2, 4, 32
    k = _bits(rng.standard_normal((1, H * d)))
    v = _bits(rng.standard_normal((1, H * d)))
    q = _bits(rng.standard_normal(Hq * d))
    out = attend_relocated(q, [{"k": k, "v": v, "delta": 77}], Hq, H, d, 1e4, 0.2)
    vv = bf16_bits_to_f64(v).reshape(H, d)
    for j in range(Hq):
        assert np.allclose(out[j * d:(j + 1) * d], vv[j // 2], atol=1e-15, rtol=0)


def test_equal_keys_average_the_values_and_a_patch_moves_them():
    """All keys equal: every weight is 1/T, so the output is the mean of V^.
    A rank-1 value patch u e_f^T adds mean(u) to feature f only."""
    rng = np.random.default_rng(63)
    T, H, Hq, d = 8, 1, 2, 4
    k = _bits(np.tile([0.5, -1.0, 0.25, 2.0], (T, 1)))
    v = _bits(rng.standard_normal((T, d)))
    q = _bits(rng.standard_normal(Hq * d))
    out = attend_relocated(q, [{"k": k, "v": v, "delta": 0}], Hq, H, d, 1e4, 1.0)
    mean = bf16_bits_to_f64(v).mean(axis=0)
    assert np.allclose(out[:d], mean, atol=1e-14, rtol=0) and np.allclose(out[d:], mean, atol=1e-14, rtol=0)
    u = np.array([[1.0], [0.5], [0.0], [2.0], [0.0], [0.0], [1.0], [0.5]])
    e = np.zeros((d, 1)); e[2, 0] = 1.0
    out2 = attend_relocated(q, [{"k": k, "v": v, "delta": 0, "uv": _bits(u), "vv": _bits(e)}], Hq, H, d, 1e4, 1.0)
    shift = np.zeros(d); shift[2] = u.mean()
    assert np.allclose(out2[:d], mean + shift, atol=1e-14, rtol=0)


def test_key_patch_changes_the_scores_as_an_added_key():
    """A key patch U_k V_k^T is the same as adding it to the keys by hand."""
    rng = np.random.default_rng(64)
    T, H, Hq, d, m = 12, 2, 2, 8, 3
    k = _bits(rng.standard_normal((T, H * d)))
    v = _bits(rng.standard_normal((T, H * d)))
    uk = _bits(rng.standard_normal((T, m)))
    vk = _bits(rng.standard_normal((H * d, m)))
    q = _bits(rng.standard_normal(Hq * d))
    got = attend_relocated(q, [{"k": k, "v": v, "delta": 0, "uk": uk, "vk": vk}], Hq, H, d, 1e4, 0.3)
    k_plus = bf16_bits_to_f64(k) + bf16_bits_to_f64(uk) @ bf16_bits_to_f64(vk).T
    want = attention(bf16_bits_to_f64(q), k_plus, bf16_bits_to_f64(v), Hq, H, d, 0.3)
    assert np.allclose(got, want, atol=1e-12, rtol=0)


def test_softmax_against_scalar_loops_and_gqa_mapping():
    rng = np.random.default_rng(65)
    T, H, Hq, d, scale = 5, 2, 6, 3, 0.7
    k = rng.standard_normal((T, H * d))
    v = rng.standard_normal((T, H * d))
    q = rng.standard_normal(Hq * d)
    got = attention(q, k, v, Hq, H, d, scale)
    g = Hq // H
    for j in range(Hq):
        h = j // g
        s = [scale * sum(q[j * d + i] * k[t, h * d + i] for i in range(d)) for t in range(T)]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        z = sum(e)
        for i in range(d):
            assert abs(got[j * d + i] - sum(e[t] / z * v[t, h * d + i] for t in range(T))) < 1e-12
    # query heads 0..2 read kv head 0, 3..5 kv head 1: swapping the kv heads swaps the output halves
    k2 = np.concatenate([k[:, d:], k[:, :d]], axis=1)
    v2 = np.concatenate([v[:, d:], v[:, :d]], axis=1)
    q2 = np.concatenate([q[g * d:], q[:g * d]])
    got2 = attention(q2, k2, v2, Hq, H, d, scale)
    assert np.allclose(np.concatenate([got2[g * d:], got2[:g * d]]), got, atol=1e-12)


def test_chunks_concatenate_along_the_context():
    rng = np.random.default_rng(66)
    H, Hq, d = 1, 1, 4
    c1 = {"k": _bits(rng.standard_normal((3, d))), "v": _bits(rng.standard_normal((3, d))), "delta": 5}
    c2 = {"k": _bits(rng.standard_normal((4, d))), "v": _bits(rng.standard_normal((4, d))), "delta": -9}
    q = _bits(rng.standard_normal(d))
    both = attend_relocated(q, [c1, c2], Hq, H, d, 1e4, 0.5)
    k1, v1 = relocated_chunk(c1["k"], c1["v"], 5, 1e4, H, d)
    k2, v2 = relocated_chunk(c2["k"], c2["v"], -9, 1e4, H, d)
    want = attention(bf16_bits_to_f64(q), np.concatenate([k1, k2]), np.concatenate([v1, v2]), Hq, H, d, 0.5)
    assert np.allclose(both, want, atol=1e-14)


def test_conditioning_sum_against_hand_values():
    """The magnitude term of the attention parity bar, sum_t p_t |v^_t| per output element
    (oracle.attend_conditioning), pinned on both sides with hand values.
    - Two tokens whose scores differ by ln 3 give weights 3/4 and 1/4.
    - Their values have opposite signs, so |sum p v| (a plausible slip) differs from
      sum p |v|.
    - Unnormalised or uniform weights differ too.
    - A rank-1 value patch that moves token 1's first element from 1 to -3 changes that
      element's term to 3/4 * 3 + 1/4 * 3."""
    from oracle import attend_conditioning
    k = _bits([[1.0, 0.0, 0.0, 0.0], [0.0, 0.0, 0.0, 0.0]])
    v = _bits([[1.0, -2.0, 0.5, 4.0], [-3.0, 2.0, 0.5, -4.0]])
    q = _bits([1.0, 0.0, 0.0, 0.0])
    scale = math.log(3.0)                       # scores ln 3 and 0
    got = attend_conditioning(q, [{"k": k, "v": v, "delta": 0}], 1, 1, 4, 1e4, scale)
    want = 0.75 * np.abs([1.0, -2.0, 0.5, 4.0]) + 0.25 * np.abs([-3.0, 2.0, 0.5, -4.0])
    assert np.allclose(got, want, rtol=1e-14, atol=0)          # [1.5, 2.0, 0.5, 4.0]
    assert not np.allclose(got, np.abs(0.75 * np.array([1.0, -2.0, 0.5, 4.0]) + 0.25 * np.array([-3.0, 2.0, 0.5, -4.0])))
    uv = _bits([[1.0], [0.0]])                  # token 1 only
    vv = _bits([[-4.0], [0.0], [0.0], [0.0]])   # feature 0 only
    got2 = attend_conditioning(q, [{"k": k, "v": v, "delta": 0, "rank": 1, "uk": None, "vk": None, "uv": uv,
                                    "vv": vv}], 1, 1, 4, 1e4, scale)
    want2 = want.copy()
    want2[0] = 0.75 * 3.0 + 0.25 * 3.0
    assert np.allclose(got2, want2, rtol=1e-14, atol=0)
