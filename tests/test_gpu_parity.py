"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element
by element, on host-drawn workloads that span several tiles and ragged tails.

Bar (the parity rule of oracle.compare): every element within 1 bf16 ulp of
the oracle rounded to bf16; with a patch (rank > 0) an element may exceed that
only as a counted mismatch inside the conditioning bound, never as a
violation; without a patch every element must be within 1 ulp; values (GQA V)
and MLA c_KV without a patch must be bit-identical to the source; slots that
no token targets must keep their sentinel bits (exact page placement)."""
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
    import position_invariant_kv_gb300 as kvrp
    kvrp.lib()


def assert_parity(reports, strict=False, limit_frac=1e-5):
    for name, r in reports.items():
        assert r["violations"] == 0, (name, r)
        if strict:
            assert r["max_ulp"] <= 1, (name, r)
        else:
            assert r["mismatches"] <= limit_frac * r["n"] + 2, (name, r)


def test_config0_single_chunk_contiguous():
    from gpu_util import run_and_compare
    wl = W.config(0)
    reps, got, want, dwl = run_and_compare(wl)
    print(reps)
    assert_parity(reps)
    assert dwl.status_value() == 0


@pytest.mark.parametrize("spec", [
    # (n_layers, n_heads, head_dim, T, delta, rank, dst_start, paged, extra_pages)
    (2, 2, 128, 200, 37, 0, 5, True, 3),          # relocation only, unaligned start, ragged tail
    (3, 4, 128, 300, -20000, 32, 0, True, 5),     # c1-like patch
    (2, 4, 64, 129, 65536, 16, 17, True, 1),      # head_dim 64, one row past a tile
    (1, 2, 128, 130, -7, 128, 3, True, 0),        # largest rank (two pipeline stages)
    (2, 1, 128, 1, 1, 64, 15, True, 2),           # a single token in the last slot of a page
    (2, 3, 128, 256, 999, 48, 0, False, 1),       # contiguous, whole tiles, rank 48
    (1, 2, 128, 77, -123, 0, 3, False, 0),        # contiguous with an offset
    (2, 8, 128, 513, 32768, 64, 31, True, 4),     # several tiles, rank 64, D = 1024
    (2, 2, 128, 131, -555, 8, 3, True, 2),        # rank 8: half of one 16-rank MMA step
    (2, 3, 64, 77, 4321, 8, 0, False, 0),         # rank 8 with head_dim 64, an odd D / 64 = 3
    (1, 4, 128, 300, 1000, 24, 5, True, 1),       # rank 24: one full step and a half
    (1, 2, 128, 140, -98765, 120, 0, True, 0),    # rank 120: the largest rank below 128
], ids=lambda s: "L{}H{}d{}T{}m{}s{}{}".format(s[0], s[1], s[2], s[3], s[5], s[6], "p" if s[7] else "c"))
def test_gqa_small(spec):
    from gpu_util import run_and_compare
    L, H, d, T, delta, m, start, paged, extra = spec
    wl = W.small_gqa(seed=100 + T + m, n_layers=L, n_heads=H, head_dim=d,
                     chunks_spec=((T, delta, m, 0),), dst_starts=[start], paged=paged, extra_pages=extra)
    reps, got, want, dwl = run_and_compare(wl)
    print(reps)
    assert_parity(reps, strict=(m == 0))
    if m == 0:
        assert np.array_equal(got["v"], want["v"])     # values copied byte for byte
    assert dwl.status_value() == 0


@pytest.mark.parametrize("rank,start,T", [(32, 0, 150), (0, 7, 150), (16, 9, 300), (8, 1, 133), (40, 0, 64)])
def test_mla_small(rank, start, T):
    from gpu_util import run_and_compare
    wl = W.small_mla(seed=300 + rank, n_layers=2, n_tokens=T, delta=-40000, rank=rank, dst_start=start,
                     extra_pages=2)
    reps, got, want, dwl = run_and_compare(wl)
    print(reps)
    assert_parity(reps, strict=(rank == 0))
    if rank == 0:
        # c_KV bytes reused unchanged
        assert np.array_equal(got["kv"][..., :512], want["kv"][..., :512])
    assert dwl.status_value() == 0


def test_batch_mixed_ranks_and_sequences():
    from gpu_util import run_and_compare
    spec = ((300, -2048, 0, 0), (150, 5000, 64, 0), (77, 0, 16, 1), (1, -1, 0, 1), (200, 31337, 32, 2),
            (256, -1024, 0, 2))
    wl = W.small_gqa(seed=400, n_layers=3, n_heads=2, head_dim=128, chunks_spec=spec, extra_pages=7,
                     dst_starts=[0, 300, 3, 80, 16, 216])
    reps, got, want, dwl = run_and_compare(wl)
    print(reps)
    assert_parity(reps)
    assert dwl.status_value() == 0


def test_batch_runs_twice_identically():
    spec = ((100, 7, 32, 0), (90, -9, 0, 0))
    wl = W.small_gqa(seed=401, n_layers=2, chunks_spec=spec)
    import harness
    dwl = harness.DeviceWorkload(wl)
    dwl.run()
    first = dwl.pools_host()
    dwl.reset_pools()
    dwl.run()
    second = dwl.pools_host()
    for n in wl.tensors:
        assert np.array_equal(first[n], second[n])


def test_patch_alone_and_strong_patch():
    """Canonical rows all zero: the output is RN(U V^T) alone; then factors at
    std 1 so that the patch dominates the rotation."""
    from gpu_util import run_and_compare
    wl = W.small_gqa(seed=500, n_layers=2, n_heads=2, head_dim=128, chunks_spec=((160, 77, 32, 0),))
    host = W.host_inputs(wl)
    for n in wl.tensors:
        host["rows"][n][:] = 0
    reps, *_ = run_and_compare(wl, host=host)
    print(reps)
    assert_parity(reps)
    host = W.host_inputs(wl)
    rng = np.random.default_rng(501)
    for n in wl.tensors:
        f = rng.standard_normal(host["u"][n][0].shape).astype(np.float32)
        host["u"][n][0] = W._f32_to_bf16_bits(f)
        f = rng.standard_normal(host["w"][n][0].shape).astype(np.float32)
        host["w"][n][0] = W._f32_to_bf16_bits(f)
    reps, *_ = run_and_compare(wl, host=host)
    print(reps)
    assert_parity(reps)


def test_empty_chunk_is_a_no_op():
    import harness
    wl = W.small_gqa(seed=600, chunks_spec=((16, 5, 16, 0),))
    host = W.host_inputs(wl)
    wl.chunks[0] = W.Chunk(0, 0, 5, 16, 0, 0)
    dwl = harness.DeviceWorkload(wl, host=host)
    dwl.run()
    torch.cuda.synchronize()
    for p in dwl.pools_host().values():
        assert np.all(p == 0xFFFF)


def test_bad_page_is_skipped_and_flagged():
    import harness
    from gpu_util import run_and_compare  # noqa: F401
    from oracle import run_workload
    wl = W.small_gqa(seed=700, n_layers=2, chunks_spec=((64, 3, 16, 0),), extra_pages=2)
    host = W.host_inputs(wl)
    good_pages = wl.block_tables.copy()
    wl.block_tables = wl.block_tables.copy()
    wl.block_tables[0, 1] = wl.num_pages + 5        # out of range: page skipped, status bit set
    dwl = harness.DeviceWorkload(wl, host=host)
    dwl.run()
    torch.cuda.synchronize()
    import position_invariant_kv_gb300 as kvrp
    assert dwl.status_value() & kvrp.KVRP_DEV_BAD_PAGE
    got = dwl.pools_host()
    wl.block_tables = good_pages
    want, _, _ = run_workload(wl, host)
    skipped = good_pages[0, 1]
    for n in wl.tensors:
        g, w_ = got[n].copy(), want[n].copy()
        assert np.all(g[:, skipped] == 0xFFFF)
        g[:, skipped] = w_[:, skipped]
        from oracle import ulp_distance
        assert ulp_distance(g, w_).max() <= 1


def test_other_stream():
    import harness
    from oracle import run_workload, ulp_distance
    wl = W.small_gqa(seed=800, n_layers=2, chunks_spec=((140, 11, 16, 0),))
    dwl = harness.DeviceWorkload(wl)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        dwl.run(stream=s)
    s.synchronize()
    got = dwl.pools_host()
    want, _, _ = run_workload(wl, dwl.host)
    for n in wl.tensors:
        assert ulp_distance(got[n], want[n]).max() <= 1


@pytest.mark.parametrize("head_dim,sections,delta,rank,T", [
    (128, (16, 24, 24), (-4537, 20000, 20000), 32, 300),   # Qwen2.5-VL layout, spatial base shift
    (128, (16, 24, 24), (12, -30000, 777), 0, 129),        # three different shifts, no patch
    (64, (8, 12, 12), (5, 6, 7), 16, 200),
    (64, (0, 16, 16), (99999, -3, 4), 0, 77),               # an empty temporal section
])
def test_mrope_small(head_dim, sections, delta, rank, T):
    from gpu_util import run_and_compare
    wl = W.small_gqa(seed=950 + T, n_layers=2, n_heads=3, head_dim=head_dim,
                     chunks_spec=((T, delta, rank, 0),), dst_starts=[9], extra_pages=2,
                     mrope_sections=sections)
    reps, got, want, dwl = run_and_compare(wl)
    print(reps)
    assert_parity(reps, strict=(rank == 0))
    assert dwl.status_value() == 0


def test_mla_batch_mixed_ranks_and_sequences():
    """kv_relocate_batch_mla: MLA chunks with their own shifts and ranks (survivors
    at rank 0, recalled chunks patched) across two sequences, in one launch."""
    from gpu_util import run_and_compare
    spec = ((150, -1024, 0, 0), (77, 31000, 32, 0), (200, -3072, 0, 1), (33, -5, 8, 1), (129, 65536, 16, 1))
    wl = W.small_mla(seed=310, n_layers=3, chunks_spec=spec, dst_start=3, extra_pages=4)
    reps, got, want, dwl = run_and_compare(wl)
    print(reps)
    assert_parity(reps)
    assert dwl.status_value() == 0
    # c_KV of the unpatched chunks is reused byte for byte
    from oracle import placement
    for c in wl.chunks:
        if c.rank == 0:
            pages, slots = placement(wl, c)
            src = dwl.host["rows"]["kv"][:, c.src_row0:c.src_row0 + c.n_tokens, :512]
            assert np.array_equal(got["kv"][:, pages, slots, :512], src)


def test_mrope_batch_video_window():
    """kv_relocate_batch_mrope: a window of video chunks, each moved by its own
    (temporal, height, width) shift, some patched, in one launch."""
    from gpu_util import run_and_compare
    spec = ((256, (-1024, 0, 0), 0, 0), (130, (-2048, 333, 333), 32, 0), (77, (4096, -7, 12), 8, 1),
            (300, (0, 0, 0), 0, 1), (64, (65000, -65000, 1), 16, 1))
    wl = W.small_gqa(seed=960, n_layers=2, n_heads=2, head_dim=128, chunks_spec=spec, extra_pages=3,
                     mrope_sections=(16, 24, 24))
    reps, got, want, dwl = run_and_compare(wl)
    print(reps)
    assert_parity(reps)
    assert dwl.status_value() == 0


def test_batch_of_many_chunks_spans_several_plan_pieces():
    """A 300-chunk batch: its launch plan is several times larger than one
    parameter-block piece, so the plan reaches the device in several copy
    launches; every chunk must still land exactly."""
    from gpu_util import run_and_compare
    spec = tuple((9 + (7 * i) % 41, (-1) ** i * (977 * i), (0, 8, 16, 0, 32)[i % 5], i % 4) for i in range(300))
    wl = W.small_gqa(seed=970, n_layers=2, n_heads=1, head_dim=128, chunks_spec=spec, extra_pages=2)
    reps, got, want, dwl = run_and_compare(wl)
    print(reps)
    assert_parity(reps)
    assert dwl.status_value() == 0


def test_launch_count_of_single_and_batch_calls():
    """kvrp_last_launch_count: one relocation launch for a single chunk; a batch
    adds the copy launches that carry its plan (31 KB each)."""
    import harness
    import position_invariant_kv_gb300 as kvrp
    one = harness.DeviceWorkload(W.small_gqa(seed=980, chunks_spec=((50, 3, 16, 0),)))
    one.run()
    assert kvrp.kvrp_last_launch_count() == 1
    spec = tuple((20, 7 * i, 16, 0) for i in range(200))
    many = harness.DeviceWorkload(W.small_gqa(seed=981, n_layers=1, n_heads=1, chunks_spec=spec))
    many.run()
    n = kvrp.kvrp_last_launch_count()
    assert 3 <= n <= 1 + -(-kvrp.kv_relocate_batch_workspace_size(200) // (31 * 1024)), n
    torch.cuda.synchronize()


def test_batch_call_captured_in_a_cuda_graph():
    """A kv_relocate_batch call recorded into a CUDA graph and replayed writes
    what the direct call writes: its plan reaches the device through kernel
    parameters, which the graph keeps, so nothing refers to host memory of the
    call after it returns."""
    import harness
    spec = ((150, -3000, 32, 0), (77, 12, 0, 0), (200, 999, 16, 1))
    wl = W.small_gqa(seed=985, n_layers=2, n_heads=2, head_dim=128, chunks_spec=spec, extra_pages=2)
    dwl = harness.DeviceWorkload(wl)
    dwl.run()
    torch.cuda.synchronize()
    want = dwl.pools_host()
    dwl.reset_pools()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dwl.run(stream=s)
    torch.cuda.synchronize()
    for _ in range(2):
        dwl.reset_pools()
        g.replay()
        torch.cuda.synchronize()
        got = dwl.pools_host()
        for n in wl.tensors:
            assert np.array_equal(got[n], want[n]), n
    assert dwl.status_value() == 0
