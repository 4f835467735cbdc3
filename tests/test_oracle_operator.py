"""Pins for the whole oracle operator KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T
(Kamera, gist.science/pt/paper/2606.23581, section 2): golden hand examples,
the family rules (values and c_KV untouched), special cases of the patch
(m = 0, X = 0, one-hot rank 1), the SVD construction of the patch
(full-rank reconstruction and the Eckart-Young residual), the conditioning
bound, and paged placement by brute force."""
import itertools
import json
import math
import os

import numpy as np
import pytest

import workloads as W
from oracle import (bf16_bits_to_f64, round_to_bf16_bits, operator_rows, row_layout, conditioning,
                    patch_product, relocate, placement, run_workload, svd_patch, eckart_young_tail)

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")))


def bits_of(vals):
    return round_to_bf16_bits(np.asarray(vals, dtype=np.float64))


def hexs(bits):
    return [f"0x{int(b):04X}" for b in np.ravel(bits)]


def test_golden_patch_order():
    g = GOLD["patch_order"]
    lay = row_layout("gqa", "k", n_heads=1, head_dim=g["head_dim"])
    ref = operator_rows(bits_of([g["x"]]), bits_of(g["u"]), bits_of(g["w"]), g["delta"], g["theta"], lay)
    assert hexs(round_to_bf16_bits(ref)) == g["expect_bits"]
    assert hexs(round_to_bf16_bits(ref)) != g["wrong_order_bits"]


def test_golden_mla():
    g = GOLD["mla"]
    lay = row_layout("mla", "kv", kv_lora_dim=g["kv_lora_dim"], rope_dim=g["rope_dim"])
    ref = operator_rows(bits_of([g["x"]]), None, None, g["delta"], g["theta"], lay)
    assert hexs(round_to_bf16_bits(ref)) == g["expect_bits"]


def test_golden_placement():
    g = GOLD["placement"]
    wl = W.Workload("t", "gqa", 1, 1, 128, 0, 128, 1e4, g["n_tokens"], 8, True,
                    [W.Chunk(0, g["n_tokens"], 0, 0, 0, g["dst_start"])],
                    np.array([g["block_table"]], np.int32))
    pages, slots = placement(wl, wl.chunks[0])
    assert list(pages) == g["expect_pages"] and list(slots) == g["expect_slots"]


def test_golden_conditioning():
    """The conditioning sum S that widens the parity bar, against hand values:
    too large an S would silently loosen every parity test, too small would
    fail them, so both sides are pinned here."""
    g = GOLD["conditioning"]
    x, u, w = bits_of([g["x"]]), bits_of(g["u"]), bits_of(g["w"])
    assert np.array_equal(bf16_bits_to_f64(x), np.array([g["x"]]))      # the hand inputs are exact in bf16
    for tensor, key in (("k", "expect_k"), ("v", "expect_v")):
        lay = row_layout("gqa", tensor, n_heads=1, head_dim=g["head_dim"])
        s = conditioning(x, u, w, g["delta"], g["theta"], lay)
        assert s.shape == (1, 4)
        np.testing.assert_allclose(s[0], g[key], rtol=1e-13, atol=0)
    # without a patch the sum keeps only the rotation terms
    lay = row_layout("gqa", "k", n_heads=1, head_dim=g["head_dim"])
    s0 = conditioning(x, None, None, g["delta"], g["theta"], lay)
    patch = np.abs(np.array(g["u"])) @ np.abs(np.array(g["w"])).T
    np.testing.assert_allclose(s0[0], np.array(g["expect_k"]) - patch[0], rtol=1e-13, atol=0)


def _rand_bits(rng, shape, std=1.0):
    return bits_of(rng.standard_normal(shape) * std)


def test_values_untouched_without_patch():
    rng = np.random.default_rng(10)
    x = _rand_bits(rng, (64, 512))
    x[0, :4] = [0x8000, 0x0000, 0x0001, 0x8001]   # signed zeros and subnormals survive
    lay = row_layout("gqa", "v", n_heads=4, head_dim=128)
    ref = operator_rows(x, None, None, 4242, 1e6, lay)
    assert np.array_equal(round_to_bf16_bits(ref), x)


def test_mla_ckv_bytes_untouched_and_rope_turned():
    rng = np.random.default_rng(11)
    x = _rand_bits(rng, (33, 576))
    lay = row_layout("mla", "kv", kv_lora_dim=512, rope_dim=64)
    ref = operator_rows(x, None, None, -54321, 1e4, lay)
    assert np.array_equal(round_to_bf16_bits(ref[:, :512]), x[:, :512])
    rope = relocate(bf16_bits_to_f64(x[:, 512:]), -54321, 1e4)
    assert np.array_equal(ref[:, 512:], rope)
    # pairs are (i, i + 32) inside the 64-dim k_rope: the 2-norm of each pair is kept
    xr = bf16_bits_to_f64(x[:, 512:])
    assert np.allclose(xr[:, :32] ** 2 + xr[:, 32:] ** 2, rope[:, :32] ** 2 + rope[:, 32:] ** 2)


def test_rank_zero_is_pure_relocation():
    rng = np.random.default_rng(12)
    x = _rand_bits(rng, (20, 256))
    lay = row_layout("gqa", "k", n_heads=2, head_dim=128)
    ref = operator_rows(x, None, None, 777, 1e6, lay)
    want = np.concatenate([relocate(bf16_bits_to_f64(x[:, :128]), 777, 1e6),
                           relocate(bf16_bits_to_f64(x[:, 128:]), 777, 1e6)], axis=1)
    assert np.array_equal(ref, want)


def test_zero_rows_give_the_patch_alone():
    rng = np.random.default_rng(13)
    u, w = _rand_bits(rng, (16, 32), 0.3), _rand_bits(rng, (256, 32), 0.3)
    x = np.zeros((16, 256), np.uint16)
    lay = row_layout("gqa", "k", n_heads=2, head_dim=128)
    ref = operator_rows(x, u, w, 999, 1e6, lay)
    uw = bf16_bits_to_f64(u) @ bf16_bits_to_f64(w).T
    assert np.array_equal(ref, uw)
    # each element equals an exactly summed dot product
    for t, f in [(0, 0), (5, 130), (15, 255)]:
        exact = math.fsum(float(a) * float(b) for a, b in zip(bf16_bits_to_f64(u[t]), bf16_bits_to_f64(w[f])))
        assert abs(ref[t, f] - exact) <= 1e-15 * max(1.0, abs(exact))


def test_one_hot_rank_one_patch_moves_one_element():
    rng = np.random.default_rng(14)
    x = _rand_bits(rng, (8, 128))
    u = np.zeros((8, 16), np.uint16)
    w = np.zeros((128, 16), np.uint16)
    u[3, 5] = bits_of(2.0)
    w[77, 5] = bits_of(0.5)
    lay = row_layout("gqa", "k", n_heads=1, head_dim=128)
    base = operator_rows(x, None, None, 5, 1e6, lay)
    ref = operator_rows(x, u, w, 5, 1e6, lay)
    diff = ref - base
    assert diff[3, 77] == 1.0
    diff[3, 77] = 0
    assert not diff.any()


@pytest.mark.parametrize("T,D,m", [(8, 16, 3), (12, 10, 5), (6, 6, 6)])
def test_svd_patch_full_rank_and_eckart_young(T, D, m):
    rng = np.random.default_rng(15)
    canon = rng.standard_normal((T, D))
    target = rng.standard_normal((T, D))             # stands for KV(B|A)
    delta = 4321
    reloc = relocate(canon, delta, 1e4)
    deficit = target - reloc
    r = min(T, D)
    U, Wm = svd_patch(deficit, r)
    assert np.allclose(reloc + U @ Wm.T, target, rtol=0, atol=1e-12)
    Um, Wmm = svd_patch(deficit, m)
    resid = np.sum((deficit - Um @ Wmm.T) ** 2)
    tail = eckart_young_tail(deficit, m)
    assert math.isclose(resid, tail, rel_tol=1e-10, abs_tol=1e-12)
    # truncation is optimal: a random rank-m perturbation of the factors does worse
    Up = Um + 1e-3 * rng.standard_normal(Um.shape)
    assert np.sum((deficit - Up @ Wmm.T) ** 2) >= resid


def test_conditioning_bounds_the_result():
    rng = np.random.default_rng(16)
    x = _rand_bits(rng, (40, 256))
    u, w = _rand_bits(rng, (40, 16), 0.05), _rand_bits(rng, (256, 16), 0.05)
    lay = row_layout("gqa", "k", n_heads=2, head_dim=128)
    ref = operator_rows(x, u, w, -31000, 1e6, lay)
    s = conditioning(x, u, w, -31000, 1e6, lay)
    assert np.all(np.abs(ref) <= s * (1 + 1e-14))


def test_patch_product_shape_and_exactness():
    rng = np.random.default_rng(17)
    u, w = _rand_bits(rng, (5, 64), 0.05), _rand_bits(rng, (7, 64), 0.05)
    p = patch_product(u, w)
    assert p.shape == (5, 7)
    for t, f in itertools.product(range(5), range(7)):
        exact = math.fsum(float(a) * float(b) for a, b in zip(bf16_bits_to_f64(u[t]), bf16_bits_to_f64(w[f])))
        assert abs(p[t, f] - exact) <= 1e-16 * 64 * max(abs(exact), 1e-3)


def _brute_force_pools(wl, inputs):
    """Element-by-element restatement: for every chunk, layer, token and
    feature, compute the output and drop it into its page slot."""
    D = wl.row_width
    pools = {n: np.full((wl.n_layers, wl.num_pages, 16, D), 0xFFFF, np.uint16) for n in wl.tensors}
    for ci, c in enumerate(wl.chunks):
        for name in wl.tensors:
            lay = row_layout(wl.family, name, n_heads=wl.n_heads, head_dim=wl.head_dim,
                             kv_lora_dim=wl.kv_lora_dim, rope_dim=wl.rope_dim)
            for l in range(wl.n_layers):
                for t in range(c.n_tokens):
                    q = c.dst_start + t
                    page = wl.block_tables[c.seq][q // 16] if wl.paged else q // 16
                    x = inputs["rows"][name][l, c.src_row0 + t][None]
                    u = inputs["u"][name][ci][l, t][None] if c.rank else None
                    w = inputs["w"][name][ci][l] if c.rank else None
                    pools[name][l, page, q % 16] = round_to_bf16_bits(
                        operator_rows(x, u, w, c.delta, wl.theta, lay))[0]
    return pools


def test_paged_placement_brute_force():
    wl = W.small_gqa(seed=20, n_layers=2, n_heads=2, head_dim=128,
                     chunks_spec=((21, 5, 16, 0), (19, -40, 0, 1), (7, 1000, 32, 0)), extra_pages=3)
    inputs = W.host_inputs(wl)
    pools, _, _ = run_workload(wl, inputs)
    brute = _brute_force_pools(wl, inputs)
    for n in wl.tensors:
        assert np.array_equal(pools[n], brute[n])
        # every targeted slot holds a value, the rest keep the sentinel
        targeted = sum(c.n_tokens for c in wl.chunks)
        written = np.any(pools[n][0] != 0xFFFF, axis=-1).sum()
        assert written == targeted


def test_block_tables_are_injective():
    for i in range(5):
        wl = W.config(i)
        if wl.block_tables is None:
            continue
        flat = wl.block_tables.ravel()
        assert len(np.unique(flat)) == flat.size
        assert flat.min() >= 0 and flat.max() < wl.num_pages
