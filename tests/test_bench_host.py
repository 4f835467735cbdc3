"""Host-side arithmetic of bench.py that needs no GPU: how a patch-formation
step is cut into concurrent calls."""
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
