"""The seeded workloads: determinism, shapes, ranges, and the algorithmic byte
counts used as the roofline numerator."""
import numpy as np
import pytest

import workloads as W

# canonical K/V read + factors read + output written, per workload
EXPECTED_BYTES = {0: 2_179_072, 1: 486_277_120, 2: 17_582_522_368, 3: 1_166_131_200, 4: 30_417_092_608}


@pytest.mark.parametrize("i", range(5))
def test_algorithmic_bytes(i):
    assert W.config(i).algorithmic_bytes()["total"] == EXPECTED_BYTES[i]


def test_config_shapes_and_ranges():
    c0 = W.config(0)
    assert c0.row_width == 1024 and c0.chunks[0].delta == 137 and c0.chunks[0].rank == 16 and not c0.paged
    c1 = W.config(1)
    assert c1.n_layers == 28 and c1.row_width == 512 and -32768 <= c1.chunks[0].delta <= 32768
    assert c1.block_tables.shape == (1, 256)
    c2 = W.config(2)
    deltas = [c.delta for c in c2.chunks]
    assert all(d % 2048 == 0 and -14336 <= d <= 14336 for d in deltas)
    assert sorted(c.dst_start for c in c2.chunks) == [k * 2048 for k in range(8)]
    assert all(c.rank == 64 for c in c2.chunks) and c2.row_width == 4096
    c3 = W.config(3)
    assert c3.family == "mla" and c3.row_width == 576 and -65536 <= c3.chunks[0].delta <= 65536
    c4 = W.config(4)
    assert len(c4.chunks) == 256
    ranks = np.array([c.rank for c in c4.chunks]).reshape(8, 32)
    assert np.all((ranks == 64).sum(axis=1) == 4) and np.all((ranks == 0).sum(axis=1) == 28)
    for c in c4.chunks:
        if c.rank == 0:
            assert c.delta % 1024 == 0 and -8 * 1024 <= c.delta <= -1024
        else:
            assert -32768 <= c.delta <= 32768


def test_host_inputs_are_deterministic():
    wl = W.small_gqa(seed=3, chunks_spec=((40, 9, 16, 0), (24, -3, 0, 0)))
    a, b = W.host_inputs(wl), W.host_inputs(wl)
    for n in wl.tensors:
        assert np.array_equal(a["rows"][n], b["rows"][n])
        assert np.array_equal(a["u"][n][0], b["u"][n][0])
        assert a["u"][n][1] is None
    assert a["rows"]["k"].shape == (wl.n_layers, 64, wl.row_width)
    assert a["u"]["k"][0].shape == (wl.n_layers, 40, 16) and a["w"]["v"][0].shape == (wl.n_layers, wl.row_width, 16)


def test_host_input_distribution():
    wl = W.small_gqa(seed=4, n_layers=1, n_heads=4, chunks_spec=((2048, 0, 32, 0),))
    x = W.host_inputs(wl)
    from oracle import bf16_bits_to_f64
    rows = bf16_bits_to_f64(x["rows"]["k"][0])
    col_std = rows.std(axis=0)
    # per-channel scales are lognormal(0, 0.5): log of column std ~ N(0, 0.5)
    assert abs(np.log(col_std).mean()) < 0.1 and 0.4 < np.log(col_std).std() < 0.6
    u = bf16_bits_to_f64(x["u"]["k"][0])
    assert abs(u.std() - 0.05) < 0.002


def test_torch_inputs_cpu_deterministic():
    wl = W.small_gqa(seed=5, chunks_spec=((30, 1, 16, 0),))
    a, b = W.torch_inputs(wl, "cpu"), W.torch_inputs(wl, "cpu")
    import torch
    assert torch.equal(a["rows"]["k"], b["rows"]["k"]) and torch.equal(a["w"]["v"][0], b["w"]["v"][0])
