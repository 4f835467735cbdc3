"""The allocation-free batch entry point, kv_relocate_batch_noalloc.

It serves callers that cannot allocate device memory (for example a plugin
that only sees tensors its host engine hands it, or a server whose memory pool
already reserved the whole GPU): instead of a caller workspace it keeps its
launch descriptors in a fixed array inside the library.  These tests call it
through the C ABI and check that it writes exactly, bit for bit, what
kv_relocate_batch writes for the same chunks, and that both agree with the
fp64 oracle:
  * on two different batches called one after the other (the second call must
    not see anything the first left in the shared array);
  * at its documented limit of KVRP_NOALLOC_MAX_CHUNKS chunks, each with its
    own sources, factors, destination pools and shift, so that the launch plan
    reaches its largest size;
  * on back-to-back calls with identical shapes whose pointers alone differ,
    so that every tensor map sits at the same place in the shared array.
The file is named so that pytest collects it last."""
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


def _noalloc(dwl, stream=None):
    import position_invariant_kv_gb300 as kvrp
    wl = dwl.wl
    kvrp.kv_relocate_batch_noalloc(dwl.batch_chunks(), n_layers=wl.n_layers, n_kv_heads=wl.n_heads,
                                   head_dim=wl.head_dim, rope_theta=wl.theta, d_status=dwl.status, stream=stream)


def _oracle_check(wl, dwl, got):
    """Every pool element against the fp64 oracle (parity rule of oracle.compare)."""
    from oracle import run_workload
    from oracle.compare import parity_report
    want, refs, conds = run_workload(wl, dwl.host)
    for name in wl.tensors:
        untouched = np.isnan(refs[name]).all(axis=-1)
        assert np.array_equal(got[name][untouched], want[name][untouched]), name
        r = parity_report(got[name][~untouched], refs[name][~untouched], conds[name][~untouched])
        assert r["violations"] == 0 and r["mismatches"] <= 1e-5 * r["n"] + 2, (name, r)


def test_noalloc_matches_workspace_batch_on_two_calls_in_a_row():
    import harness
    first = W.small_gqa(seed=900, n_layers=3, n_heads=2, head_dim=128,
                        chunks_spec=((300, -2048, 0, 0), (150, 5000, 64, 0), (77, 0, 16, 1), (200, 31337, 32, 1)),
                        dst_starts=[0, 300, 5, 90], extra_pages=3)
    # a second, larger batch with other shifts, ranks, head size and layout
    spec = tuple((64 + 37 * (i % 5), (-1) ** i * 1024 * (i % 7), (0, 16, 0, 8, 32, 0, 64)[i % 7], i % 3)
                 for i in range(40))
    second = W.small_gqa(seed=901, n_layers=2, n_heads=4, head_dim=64, chunks_spec=spec, extra_pages=5)
    for wl in (first, second):
        dwl = harness.DeviceWorkload(wl)
        dwl.run()                                   # kv_relocate_batch with a torch workspace
        torch.cuda.synchronize()
        want = dwl.pools_host()
        dwl.reset_pools()
        dwl.status.zero_()
        _noalloc(dwl)
        torch.cuda.synchronize()
        got = dwl.pools_host()
        assert dwl.status_value() == 0
        for name in wl.tensors:
            assert np.array_equal(got[name], want[name]), name
        _oracle_check(wl, dwl, got)


def test_noalloc_at_its_chunk_limit_with_distinct_maps():
    """KVRP_NOALLOC_MAX_CHUNKS chunks, every one patched, with its own shift and
    its own destination pools (half of them paged through a block table of
    their own): eight distinct tensor maps and one phase table per chunk."""
    import harness
    import position_invariant_kv_gb300 as kvrp
    from gpu_util import bits
    from oracle import chunk_layer_rows
    from oracle.compare import parity_report
    n = kvrp.KVRP_NOALLOC_MAX_CHUNKS
    spec = tuple((3 + (5 * i) % 29, 7919 * i - 1000003, (8, 16, 24, 32)[i % 4], 0) for i in range(n))
    wl = W.small_gqa(seed=910, n_layers=2, n_heads=1, head_dim=64, chunks_spec=spec, paged=False)
    dwl = harness.DeviceWorkload(wl)
    D, L = wl.row_width, wl.n_layers
    g = torch.Generator().manual_seed(911)
    pools, tables, chunks = [], [], []
    for ci, c in enumerate(wl.chunks):
        start = ci % 16
        n_pages = (start + c.n_tokens + 15) // 16 + 1
        ps = {t: torch.empty((L, n_pages, 16, D), dtype=torch.bfloat16, device="cuda") for t in wl.tensors}
        bt = torch.randperm(n_pages, generator=g).to(torch.int32).cuda() if ci % 2 else None
        dsts = [kvrp.Dst(base=ps[t], num_pages=n_pages, layer_stride=ps[t].stride(0), block_table=bt,
                         dst_start=start) for t in wl.tensors]
        pools.append(ps)
        tables.append(bt)
        chunks.append(kvrp.Chunk(k_src=dwl._src("k", c), v_src=dwl._src("v", c), n_tokens=c.n_tokens,
                                 delta=c.delta, k_dst=dsts[0], v_dst=dsts[1], rank=c.rank,
                                 uk=dwl.u["k"][ci], vk=dwl.w["k"][ci], uv=dwl.u["v"][ci], vv=dwl.w["v"][ci],
                                 src_layer_stride=dwl.rows["k"].stride(0), u_layer_stride=c.n_tokens * c.rank,
                                 v_layer_stride=D * c.rank))

    def reset():
        for ps in pools:
            for p in ps.values():
                p.view(torch.int16).fill_(-1)

    ws = torch.empty(kvrp.kv_relocate_batch_workspace_size(n), dtype=torch.uint8, device="cuda")
    reset()
    kvrp.kv_relocate_batch(chunks, n_layers=L, n_kv_heads=wl.n_heads, head_dim=wl.head_dim, rope_theta=wl.theta,
                           workspace=ws, d_status=dwl.status)
    torch.cuda.synchronize()
    want = [{t: bits(p) for t, p in ps.items()} for ps in pools]
    reset()
    kvrp.kv_relocate_batch_noalloc(chunks, n_layers=L, n_kv_heads=wl.n_heads, head_dim=wl.head_dim,
                                   rope_theta=wl.theta, d_status=dwl.status)
    torch.cuda.synchronize()
    assert dwl.status_value() == 0
    report = {}
    for ci, c in enumerate(wl.chunks):
        start = ci % 16
        q = start + np.arange(c.n_tokens)
        bt = None if tables[ci] is None else tables[ci].cpu().numpy()
        page = q // 16 if bt is None else bt[q // 16]
        for t, p in pools[ci].items():
            got = bits(p)
            assert np.array_equal(got, want[ci][t]), (ci, t)
            hit = np.zeros(got.shape[1:3], bool)
            hit[page, q % 16] = True
            assert np.all(got[:, ~hit] == 0xFFFF), (ci, t)       # nothing outside the chunk's slots
            for l in range(L):
                ref, cond = chunk_layer_rows(wl, dwl.host, ci, t, l)
                r = parity_report(got[l, page, q % 16], ref, cond)
                report = {k: report.get(k, 0) + v if not k.startswith("max") else max(report.get(k, 0), v)
                          for k, v in r.items()}
    print(report)
    assert report["violations"] == 0 and report["mismatches"] <= 1e-5 * report["n"] + 2, report


def test_noalloc_same_shapes_new_pointers_back_to_back():
    """Two batches with identical shapes and different pointers and data, called
    alternately on one stream with no synchronisation in between: each result
    must be its own batch's, bit for bit."""
    import harness
    spec = ((130, -4096, 32, 0), (60, 777, 0, 0), (200, -1, 16, 1), (17, 5, 8, 1))
    sets = []
    for seed in (920, 921):
        wl = W.small_gqa(seed=seed, n_layers=2, n_heads=2, head_dim=128, chunks_spec=spec, extra_pages=2)
        dwl = harness.DeviceWorkload(wl)
        dwl.run()
        torch.cuda.synchronize()
        sets.append((wl, dwl, dwl.pools_host()))
    for order in ((0, 1, 0, 1), (1, 0, 1, 0)):
        for _, dwl, _ in sets:
            dwl.reset_pools()
            dwl.status.zero_()
        for i in order:
            _noalloc(sets[i][1])
        torch.cuda.synchronize()
        for wl, dwl, want in sets:
            got = dwl.pools_host()
            assert dwl.status_value() == 0
            for name in wl.tensors:
                assert np.array_equal(got[name], want[name]), (order, name)
    wl, dwl, _ = sets[1]
    _oracle_check(wl, dwl, dwl.pools_host())


def test_noalloc_rejects_batches_over_its_limit():
    import position_invariant_kv_gb300 as kvrp
    d = kvrp.Dst(base=0x10000, num_pages=4)
    ch = kvrp.Chunk(k_src=0x20000, v_src=0x30000, n_tokens=10, delta=3, k_dst=d, v_dst=d)
    with pytest.raises(kvrp.KvrpError) as e:
        kvrp.kv_relocate_batch_noalloc([ch] * (kvrp.KVRP_NOALLOC_MAX_CHUNKS + 1), n_layers=1, n_kv_heads=2,
                                       head_dim=128, rope_theta=1e4, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_INVALID_ARG
    assert "at most" in str(e.value)
