"""GPU decode attention over relocated, patched chunks (kv_attend_relocated)
against the fp64 oracle, element by element.

The oracle materialises K^ = R(delta) K + U_k V_k^T and V^ = V + U_v V_v^T of
every chunk in fp64 and evaluates softmax(scale q K^T) V^ (Kamera,
gist.science/pt/paper/2606.23581, section 2, read side).  The kernel never
forms K^ or V^: it rotates the query by R(-delta) and adds the rank-m terms.
The bar: within 1 bf16 ulp of the oracle rounded once to bf16; an element off
by more must still lie within ulp(ref) + 2^-14 * sum_t p_t |v^_t| (the fp32
rounding of the scores and sums, bounded by that magnitude)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from position_invariant_kv_gb300.build import build
    build()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make_case(seed, seqs, Hq, Hkv, d):
    """seqs: list of sequences, each a list of (n_tokens, rank) chunks.  Inputs
    are seeded normal draws (fp32) rounded to bf16 (nearest even), as bits."""
    rng = np.random.default_rng(seed)
    D = Hkv * d

    def bf16(shape, std=1.0):
        x = torch.from_numpy((std * rng.standard_normal(shape, dtype=np.float32)).astype(np.float32))
        return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    q = bf16((len(seqs), Hq, d))
    chunks, seq_chunks = [], [0]
    for s in seqs:
        for (T, m) in s:
            c = {"k": bf16((T, D)), "v": bf16((T, D)), "delta": int(rng.integers(-40000, 40001)), "rank": m}
            if m:
                c["uk"], c["vk"] = bf16((T, m), 0.3), bf16((D, m), 0.1)
                c["uv"], c["vv"] = bf16((T, m), 0.3), bf16((D, m), 0.1)
            chunks.append(c)
        seq_chunks.append(len(chunks))
    return q, chunks, seq_chunks


def paged_pool(rows, seed):
    """rows [T][D] bf16 bits placed in a pool of 16-token pages: the chunk's pages
    shuffled among 3 more pages than it needs, the unused ones NaN.  Returns the
    pool [pages][16][D], the block table and the page count."""
    T, D = rows.shape
    need = (T + 15) // 16
    n_pages = need + 3
    table = np.random.default_rng(seed).permutation(n_pages)[:need].astype(np.int32)
    pool = np.full((n_pages, 16, D), 0x7FC0, dtype=np.uint16)
    for t in range(T):
        pool[table[t // 16], t % 16] = rows[t]
    return pool, table, n_pages


def run_gpu(q, chunks, seq_chunks, Hq, Hkv, d, theta, scale, paged=False, status_ok=True):
    import position_invariant_kv_gb300 as kvrp
    keep = []
    ac = []
    for i, c in enumerate(chunks):
        T = c["k"].shape[0]
        f = [(_dev(c[n]) if c["rank"] else None) for n in ("uk", "vk", "uv", "vv")]
        if paged and T:
            pk, table, n_pages = paged_pool(c["k"], 100 + i)
            pv, _, _ = paged_pool(c["v"], 100 + i)
            k, v = _dev(pk), _dev(pv)
            tab = torch.from_numpy(c.get("table_override", table)).cuda()
            keep += [tab]
            extra = dict(block_table=tab, num_pages=n_pages)
        else:
            k = _dev(c["k"]) if T else torch.empty((16,), dtype=torch.bfloat16, device="cuda")
            v = _dev(c["v"]) if T else torch.empty((16,), dtype=torch.bfloat16, device="cuda")
            extra = {}
        keep += [k, v] + f
        ac.append(kvrp.AttnChunk(k=k, v=v, n_tokens=T, delta=c["delta"], rank=c["rank"], uk=f[0], vk=f[1], uv=f[2],
                                 vv=f[3], **extra))
    out = torch.empty((len(seq_chunks) - 1, Hq, d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(kvrp.kv_attend_relocated_workspace_size([c["k"].shape[0] for c in chunks], Hq, Hkv, d),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvrp.kv_attend_relocated(_dev(q), ac, seq_chunks, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, rope_theta=theta,
                             softmax_scale=scale, out=out, workspace=ws, d_status=status)
    torch.cuda.synchronize()
    if status_ok:
        assert int(status.item()) == 0
        return _bits(out)
    return _bits(out), int(status.item())


def check(got, q, chunks, seq_chunks, Hq, Hkv, d, theta, scale):
    from oracle import attend_conditioning, attend_relocated, bf16_bits_to_f64, bf16_ulp, round_to_bf16_bits
    from oracle.bf16 import ulp_distance
    worst = 0
    for s in range(len(seq_chunks) - 1):
        cs = [dict(c, **({} if c["rank"] else {"uk": None, "vk": None, "uv": None, "vv": None}))
              for c in chunks[seq_chunks[s]:seq_chunks[s + 1]] if c["k"].shape[0] > 0]
        g = got[s].reshape(-1)
        if not cs:
            assert np.all(bf16_bits_to_f64(g) == 0.0)
            continue
        ref = attend_relocated(q[s].reshape(-1), cs, Hq, Hkv, d, theta, scale)
        cond = attend_conditioning(q[s].reshape(-1), cs, Hq, Hkv, d, theta, scale)
        dist = ulp_distance(g, round_to_bf16_bits(ref))
        err = np.abs(bf16_bits_to_f64(g) - ref)
        bound = bf16_ulp(ref) + 2.0 ** -14 * cond
        assert np.all((dist <= 1) | (err <= bound)), (s, int(dist.max()), float((err / bound).max()))
        worst = max(worst, int(dist.max()))
    return worst


@pytest.mark.parametrize("seqs,Hq,Hkv,d", [
    ([[(300, 32), (77, 0)], [(1, 0)], [(128, 16), (129, 32), (513, 16)]], 28, 4, 128),   # GQA, ragged, mixed ranks
    ([[(200, 16), (64, 16)], [(1000, 32)]], 8, 8, 64),                                    # MHA, head_dim 64
    ([[(260, 32)], [(17, 0), (300, 16)]], 32, 2, 128),                                    # 16 query heads per KV head
    ([[(100, 48), (50, 128)], [(65, 0), (1, 128)]], 6, 3, 64),                            # odd KV heads; ranks 48, 128
    ([[(9000, 32), (7000, 16)], [(12000, 0)]], 16, 4, 128),                               # long: several stages per CTA
    ([[(300, 64), (129, 128)], [(77, 96)]], 28, 4, 128),                                   # ranks above 32 at head_dim 128
    ([[(200, 128), (33, 64)], [(150, 0)]], 32, 2, 128),                                    # 16 heads per KV head, rank 128
    # ~16-stage shares on 152 SMs, chunks starting inside shares (mid-share segment changes)
    ([[(19000, 16), (23000, 32)], [(17000, 0), (21000, 16)]], 8, 4, 64),
])
def test_attention_matches_oracle(seqs, Hq, Hkv, d):
    import position_invariant_kv_gb300 as kvrp
    theta, scale = 1e6, d ** -0.5
    q, chunks, sc = make_case(7 + Hq, seqs, Hq, Hkv, d)
    got = run_gpu(q, chunks, sc, Hq, Hkv, d, theta, scale)
    assert kvrp.kvrp_last_launch_count() == 2   # block and combine kernels
    worst = check(got, q, chunks, sc, Hq, Hkv, d, theta, scale)
    print("worst ulp distance", worst)
    # the same chunks read from paged pools (shuffled pages, unused pages NaN): the same bits
    paged = run_gpu(q, chunks, sc, Hq, Hkv, d, theta, scale, paged=True)
    assert np.array_equal(paged, got)


def test_bad_page_is_flagged_not_faulted():
    """A block-table entry outside the pool sets KVRP_DEV_BAD_PAGE; the kernel reads
    page 0 instead of faulting, and the other sequence is untouched."""
    import position_invariant_kv_gb300 as kvrp
    Hq, Hkv, d, theta, scale = 8, 4, 128, 1e6, 0.088
    q, chunks, sc = make_case(93, [[(100, 16)], [(64, 0)]], Hq, Hkv, d)
    good = run_gpu(q, chunks, sc, Hq, Hkv, d, theta, scale, paged=True)
    _, table, n_pages = paged_pool(chunks[0]["k"], 100)
    bad = table.copy()
    bad[3] = n_pages + 5
    chunks[0]["table_override"] = bad
    got, status = run_gpu(q, chunks, sc, Hq, Hkv, d, theta, scale, paged=True, status_ok=False)
    assert status & kvrp.KVRP_DEV_BAD_PAGE
    assert np.array_equal(got[1], good[1])


def test_empty_sequences_and_chunks():
    """A sequence with no chunks and one whose only chunk is empty get zeros;
    an empty chunk between two others changes nothing."""
    Hq, Hkv, d, theta, scale = 4, 2, 64, 1e4, 0.125
    q, chunks, sc = make_case(91, [[(50, 16), (0, 0), (40, 0)], [], [(0, 0)]], Hq, Hkv, d)
    got = run_gpu(q, chunks, sc, Hq, Hkv, d, theta, scale)
    check(got, q, chunks, sc, Hq, Hkv, d, theta, scale)


def test_shift_moves_only_through_the_rotation():
    """delta = 0 and no patch: plain attention over the canonical cache; the
    same chunk with delta != 0 differs (the relocation is applied)."""
    from oracle import attention, bf16_bits_to_f64, round_to_bf16_bits
    Hq, Hkv, d = 4, 2, 128
    q, chunks, sc = make_case(92, [[(100, 0)]], Hq, Hkv, d)
    chunks[0]["delta"] = 0
    got0 = run_gpu(q, chunks, sc, Hq, Hkv, d, 1e4, 0.088)
    ref0 = attention(bf16_bits_to_f64(q[0].reshape(-1)), bf16_bits_to_f64(chunks[0]["k"]),
                     bf16_bits_to_f64(chunks[0]["v"]), Hq, Hkv, d, 0.088)
    from oracle.bf16 import ulp_distance
    assert ulp_distance(got0[0].reshape(-1), round_to_bf16_bits(ref0)).max() <= 1
    chunks[0]["delta"] = 5000
    got1 = run_gpu(q, chunks, sc, Hq, Hkv, d, 1e4, 0.088)
    assert np.any(got1 != got0)


def test_bench_workload_on_sampled_sequences():
    """The bench's own workload and launch (16 sequences x 4 chunks x 4096 tokens,
    28 query / 4 KV heads x 128, rank-32 K and V patches, canonical K and V in a
    shuffled paged pool): sequences 0, 7 and 15 against the oracle, every output
    element of each (the oracle gets each chunk's rows gathered through its table)."""
    import bench
    import position_invariant_kv_gb300 as kvrp
    a = dict(bench.ATTN_SHAPE)
    keep, chunks, q, sc = bench.attend_workload(a, "cuda")
    out = torch.empty_like(q)
    ws = torch.empty(kvrp.kv_attend_relocated_workspace_size([c.n_tokens for c in chunks], a["Hq"], a["Hkv"], a["d"]),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = a["d"] ** -0.5
    kvrp.kv_attend_relocated(q, chunks, sc, n_q_heads=a["Hq"], n_kv_heads=a["Hkv"], head_dim=a["d"],
                             rope_theta=a["theta"], softmax_scale=scale, out=out, workspace=ws, d_status=status)
    assert kvrp.kvrp_last_launch_count() == 2   # block and combine kernels
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = _bits(out)
    qb = _bits(q)
    pool_k, pool_v = _bits(chunks[0].k), _bits(chunks[0].v)   # the shared paged pools [pages][16][D]

    def rows(pool, c):   # the chunk's rows, gathered through its block table
        table = c.block_table.cpu().numpy()
        t = np.arange(c.n_tokens)
        return pool[table[t // 16], t % 16]

    for s in (0, 7, 15):
        host = [{"k": rows(pool_k, c), "v": rows(pool_v, c), "delta": c.delta, "rank": c.rank, "uk": _bits(c.uk),
                 "vk": _bits(c.vk), "uv": _bits(c.uv), "vv": _bits(c.vv)} for c in chunks[sc[s]:sc[s + 1]]]
        sub_sc = [0, len(host)]
        worst = check(got[s:s + 1], qb[s:s + 1], host, sub_sc, a["Hq"], a["Hkv"], a["d"], a["theta"], scale)
        print("sequence", s, "worst ulp distance", worst)


def test_many_chunks_and_sequences():
    """200 chunks (1 to 90 tokens, mixed ranks) over 50 sequences: the parameter block
    near its limit and partial lists that cross many CTA shares."""
    rng = np.random.default_rng(95)
    seqs, n = [], 0
    while n < 200:
        k = int(min(rng.integers(1, 8), 200 - n))
        seqs.append([(int(rng.integers(1, 91)), int(rng.choice([0, 16, 32]))) for _ in range(k)])
        n += k
    Hq, Hkv, d, theta, scale = 8, 2, 128, 1e6, 128 ** -0.5
    q, chunks, sc = make_case(96, seqs, Hq, Hkv, d)
    got = run_gpu(q, chunks, sc, Hq, Hkv, d, theta, scale)
    worst = check(got, q, chunks, sc, Hq, Hkv, d, theta, scale)
    print(len(seqs), "sequences, worst ulp distance", worst)
