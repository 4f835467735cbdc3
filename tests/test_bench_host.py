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
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
