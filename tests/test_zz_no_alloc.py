"""The allocation-free batch entry point, kv_relocate_batch_noalloc.

It serves callers that cannot allocate device memory (for example a plugin
that only sees tensors its host engine hands it, or a server whose memory pool
already reserved the whole GPU): instead of a caller workspace it keeps its
launch descriptors in a fixed array inside the library.  These tests call it
through the C ABI and check that it writes exactly what kv_relocate_batch
writes for the same chunks, on two different batches called one after the
other (the second call must not see anything the first left in the shared
array).  The file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from position_invariant_kv_gb300.build import build
    build()


def _batch_pair(wl):
    """(pools from kv_relocate_batch, pools from kv_relocate_batch_noalloc, status)."""
    import harness
    import position_invariant_kv_gb300 as kvrp
    dwl = harness.DeviceWorkload(wl)
    dwl.run()                                   # kv_relocate_batch with a torch workspace
    torch.cuda.synchronize()
    want = dwl.pools_host()
    dwl.reset_pools()
    dwl.status.zero_()
    kvrp.kv_relocate_batch_noalloc(dwl.batch_chunks(), n_layers=wl.n_layers, n_kv_heads=wl.n_heads,
                                   head_dim=wl.head_dim, rope_theta=wl.theta, d_status=dwl.status)
    torch.cuda.synchronize()
    return want, dwl.pools_host(), dwl.status_value()


def _same_within_tolerance(got, want):
    from oracle import ulp_distance
    untouched = want == 0xFFFF
    assert np.array_equal(got[untouched], want[untouched])          # placement is exact
    assert ulp_distance(got[~untouched], want[~untouched]).max() <= 1


def test_noalloc_matches_workspace_batch_on_two_calls_in_a_row():
    first = W.small_gqa(seed=900, n_layers=3, n_heads=2, head_dim=128,
                        chunks_spec=((300, -2048, 0, 0), (150, 5000, 64, 0), (77, 0, 16, 1), (200, 31337, 32, 1)),
                        dst_starts=[0, 300, 5, 90], extra_pages=3)
    # a second, larger batch with other shifts, ranks, head size and layout
    spec = tuple((64 + 37 * (i % 5), (-1) ** i * 1024 * (i % 7), (0, 16, 0, 32, 0, 64)[i % 6], i % 3)
                 for i in range(40))
    second = W.small_gqa(seed=901, n_layers=2, n_heads=4, head_dim=64, chunks_spec=spec, extra_pages=5)
    for wl in (first, second):
        want, got, status = _batch_pair(wl)
        assert status == 0
        for name in wl.tensors:
            _same_within_tolerance(got[name], want[name])


def test_noalloc_rejects_batches_over_its_limit():
    import position_invariant_kv_gb300 as kvrp
    d = kvrp.Dst(base=0x10000, num_pages=4)
    ch = kvrp.Chunk(k_src=0x20000, v_src=0x30000, n_tokens=10, delta=3, k_dst=d, v_dst=d)
    with pytest.raises(kvrp.KvrpError) as e:
        kvrp.kv_relocate_batch_noalloc([ch] * (kvrp.KVRP_NOALLOC_MAX_CHUNKS + 1), n_layers=1, n_kv_heads=2,
                                       head_dim=128, rope_theta=1e4, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_INVALID_ARG
    assert "at most" in str(e.value)
