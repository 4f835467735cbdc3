"""Pins for the two acceptance helpers the GPU tests decide with: the parity
rule of oracle.compare (within 1 bf16 ulp of the fp64 result rounded to bf16,
or a counted mismatch inside the conditioned bound) and the attention
conditioning sum of oracle.attend (sum over tokens of p_t |V^_t|).  They are
checked on hand-built cases whose outcome is fixed by the definitions: exact
grid values, neighbours one and two ulps away, and attention inputs whose
values make the sum a closed form."""
import numpy as np

from oracle import attend_conditioning, attend_relocated, bf16_bits_to_f64, round_to_bf16_bits
from oracle.compare import COND_FACTOR, parity_report


def _bits(x):
    return round_to_bf16_bits(np.asarray(x, dtype=np.float64))


def test_parity_rule_on_hand_cases():
    # 1.0 has bits 0x3F80; its bf16 neighbours above are 0x3F81 (1 + 2^-7) and 0x3F82
    ref = np.array([1.0, 1.0, 1.0, 1.0, -3.0])
    got = np.array([0x3F80, 0x3F81, 0x3F82, 0x3F7F, 0xC040], dtype=np.uint16)   # last: -3.0 exactly
    rep = parity_report(got, ref, np.zeros(5))
    assert rep["n"] == 5
    assert (rep["ulp0"], rep["ulp1"], rep["mismatches"]) == (2, 2, 1)
    assert rep["max_ulp"] == 2
    # two ulps off with no conditioning slack is outside the bound
    assert rep["violations"] == 1
    assert np.isclose(rep["max_rel_err"], 2.0 ** -6)


def test_conditioned_bound_admits_a_cancelled_element():
    """A value that nearly cancels (|ref| tiny against the terms that formed it)
    may miss by more than an ulp of ref: a mismatch, not a violation, while the
    error stays within ulp(ref) + 2^-20 * cond."""
    ref = np.array([1e-6])
    want = _bits(ref)[0]
    off = np.uint16(want + 3)                                  # three ulps away
    err = abs(bf16_bits_to_f64(np.array([off]))[0] - ref[0])
    small = parity_report(np.array([off]), ref, np.array([0.0]))
    large = parity_report(np.array([off]), ref, np.array([2.0 * err / COND_FACTOR]))
    assert small["mismatches"] == 1 and small["violations"] == 1
    assert large["mismatches"] == 1 and large["violations"] == 0


def test_signed_zero_and_exact_results_pass():
    ref = np.array([0.0, -0.0, 0.5])
    got = np.array([0x8000, 0x0000, 0x3F00], dtype=np.uint16)   # -0, +0, 0.5
    rep = parity_report(got, ref, np.zeros(3))
    assert rep["ulp0"] == 3 and rep["mismatches"] == 0 and rep["max_rel_err"] == 0.0


def _chunks(rng, T, D, v_sign=None):
    v = rng.standard_normal((T, D))
    if v_sign == "pos":
        v = np.abs(v)
    return [{"k": _bits(rng.standard_normal((T, D))), "v": _bits(v), "delta": int(rng.integers(-500, 500))}]


def test_conditioning_equals_the_output_for_nonnegative_values():
    """With every V^ entry >= 0 (no patch), sum_t p_t |V^_t| is the attention
    output itself, head mapping included."""
    rng = np.random.default_rng(81)
    Hq, H, d, T = 6, 2, 16, 23
    cs = _chunks(rng, T, H * d, "pos") + _chunks(rng, 9, H * d, "pos")
    q = _bits(rng.standard_normal(Hq * d))
    out = attend_relocated(q, cs, Hq, H, d, 1e4, 0.3)
    cond = attend_conditioning(q, cs, Hq, H, d, 1e4, 0.3)
    assert np.allclose(cond, out, rtol=1e-12, atol=0)


def test_conditioning_bounds_the_output_and_is_exact_for_one_token():
    rng = np.random.default_rng(82)
    Hq, H, d = 4, 2, 8
    cs = _chunks(rng, 31, H * d)
    q = _bits(rng.standard_normal(Hq * d))
    out = attend_relocated(q, cs, Hq, H, d, 1e4, 0.25)
    cond = attend_conditioning(q, cs, Hq, H, d, 1e4, 0.25)
    assert np.all(cond >= np.abs(out) - 1e-12)
    assert np.any(cond > np.abs(out) + 1e-3)                   # mixed signs: a strict bound somewhere
    one = _chunks(rng, 1, H * d)
    c1 = attend_conditioning(q, one, Hq, H, d, 1e4, 0.25).reshape(Hq, d)
    v = np.abs(bf16_bits_to_f64(one[0]["v"])).reshape(H, d)
    for j in range(Hq):
        assert np.allclose(c1[j], v[j // (Hq // H)], rtol=0, atol=1e-15)
