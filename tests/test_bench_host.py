"""Host-side parts of bench.py that need no GPU: how a patch-formation step
is cut into concurrent calls, and the reference arm's JSON line."""
import pytest

import bench


@pytest.mark.parametrize("tensors,L,streams", [
    (("k", "v"), 28, 1), (("k", "v"), 28, 2), (("k", "v"), 28, 4), (("k", "v"), 28, 8),
    (("kv",), 60, 4), (("kv",), 3, 8), (("k", "v"), 1, 16), (("k", "v"), 31, 6),
])
def test_patch_form_jobs_cover_every_layer_once(tensors, L, streams):
    jobs, per = bench.patch_form_jobs(tensors, L, streams)
    assert per == max(1, streams // len(tensors))
    for n in tensors:
        ranges = sorted((l0, l1) for (t, l0, l1) in jobs if t == n)
        assert all(l1 > l0 for l0, l1 in ranges)                       # no empty call
        covered = [l for l0, l1 in ranges for l in range(l0, l1)]
        assert covered == list(range(L))                                # every layer once, in order
        sizes = [l1 - l0 for l0, l1 in ranges]
        assert max(sizes) - min(sizes) <= 1                             # nearly equal ranges
        assert len(ranges) == min(per, L)
    assert len(jobs) <= max(streams, len(tensors))


def test_one_stream_runs_whole_tensors():
    jobs, per = bench.patch_form_jobs(("k", "v"), 28, 1)
    assert per == 1 and jobs == [("k", 0, 28), ("v", 0, 28)]


def test_reference_arm_line_contract():
    """The reference arm's JSON line (the fp64 oracle on host cores) carries the
    keys of the bench contract, names our arm's metric and workload, and marks
    itself with impl, a cpu_baseline and an e2e without host-device bytes."""
    class Args:
        config, steps, warmup = 1, 2, 0
    line = bench.bench_reference(Args())
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in line, key
    assert line["metric"] == bench.METRIC and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["impl"] == "reference" and line["steps"] == 2 and line["value"] > 0
    assert line["config"]["workload"].startswith("c1_")
    import workloads as W
    assert line["config"] == bench.bench_config(W.config(1), 1)      # the same config object as our arm's
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"] and cb["sample"]
    assert cb["os_cpu_count"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_oracle_sampler_weights_the_chunk_kinds_of_the_window_batch():
    """c4 mixes 224 unpatched and 32 rank-64 chunks: the CPU baseline samples one
    chunk of each kind, in proportion to their tokens."""
    o = bench.OracleSampler(4)
    ranks = [c.rank for c in o.slice_wl.chunks]
    assert sorted(ranks) == [0, 64]
    share = dict(zip(ranks, o.share))
    assert share[0] == pytest.approx(224 / 256) and share[64] == pytest.approx(32 / 256)
    secs, rows = o.step(64)
    assert secs > 0 and rows == 56 + 8


def test_parity_worker_reports_the_sampled_rows(tmp_path):
    """The bench's in-run parity check: rows the oracle itself rounds pass with
    no mismatch, and a row moved by 3 ulp counts as a mismatch and, outside the
    conditioning bound, as a violation."""
    import pickle
    import numpy as np
    import workloads as W
    from oracle import operator_rows, round_to_bf16_bits, row_layout
    wl = W.small_gqa(seed=5, n_layers=1, n_heads=2, head_dim=128, chunks_spec=((8, 1000, 16, 0),))
    host = W.host_inputs(wl)
    x, u, w = host["rows"]["k"][0], host["u"]["k"][0][0], host["w"]["k"][0][0]
    ref = operator_rows(x, u, w, 1000, wl.theta, row_layout("gqa", "k", n_heads=2, head_dim=128))
    got = round_to_bf16_bits(ref)
    g = {"family": "gqa", "tensor": "k", "n_heads": 2, "head_dim": 128, "kv_lora_dim": 0, "rope_dim": 128,
         "delta": 1000, "theta": wl.theta, "sections": None, "x": x, "u": u, "w": w, "got": got}
    path = tmp_path / "s.pkl"
    path.write_bytes(pickle.dumps([g]))
    r = bench.parity_worker(str(path))
    assert r["rows"] == 8 and r["n"] == 8 * 256 and r["mismatches"] == 0 and r["violations"] == 0
    bad = got.copy()
    big = np.argmax(np.abs(ref).ravel())
    bad.ravel()[big] += 3
    g["got"] = bad
    path.write_bytes(pickle.dumps([g]))
    r = bench.parity_worker(str(path))
    assert r["mismatches"] == 1 and r["violations"] == 1 and r["max_ulp"] == 3


def test_e2e_leg_fits_host_memory():
    """The end-to-end leg moves every layer when the pinned buffers fit, and
    fewer (at least one) when they would not."""
    import workloads as W
    wl = W.config(4)
    per_layer = (wl.algorithmic_bytes()["total"] + wl.n_layers * wl.num_pages * 16 * wl.row_width * 2 * 2) / wl.n_layers
    assert bench.e2e_layers(wl, 1 << 62) == wl.n_layers
    assert bench.e2e_layers(wl, int(per_layer * 10.5)) == 10
    assert bench.e2e_layers(wl, 1) == 1
    assert bench.host_budget_bytes() > 0


def test_method_bytes_of_patch_formation_and_attention():
    """The bytes the roofline fractions divide by, counted by hand for small shapes.
    Patch formation, per tensor: the caches read once (the conditioned ones orbit times),
    the bf16 deficit written twice, read by each of the 2q + 3 tensor-core passes, each
    pass's fp32 output, the Gram's and the apply's reads in each of the 2q + 2
    orthonormalisation rounds, and the bf16 factors.  Decode attention: every chunk's K,
    V and factor rows, V_k and V_v, and the queries in and the output out."""
    import bench
    L, T, D, m, p, q, orbit = 2, 100, 64, 16, 8, 1, 1
    kp = 32                                     # m + p padded to 16
    n = L * T * D
    skinny = L * (T + D) * kp * 4
    want = (2 * n * 2                           # canonical and one conditioned cache, bf16
            + 2 * n * 2                         # the deficit written as rows and as transposed rows
            + 5 * n * 2                         # 2q + 3 passes read it
            + 5 * skinny                        # each pass writes its fp32 output
            + 4 * 2 * skinny                    # 2q + 2 rounds: the Gram's and the apply's reads
            + L * (T + D) * m * 2)              # the factors U, V in bf16
    assert bench.patch_bytes(L, T, D, m, p, q, orbit) == want
    a = dict(seqs=2, chunks=3, tokens=100, Hq=8, Hkv=2, d=64, rank=16)
    per_chunk = 100 * 128 * 2 * 2 + 100 * 16 * 2 * 2 + 128 * 16 * 2 * 2
    assert bench.attn_bytes(a) == 6 * per_chunk + 2 * 8 * 64 * 2 * 2
