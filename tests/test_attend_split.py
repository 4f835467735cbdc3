"""Host-side planning of the decode-attention call, through the testing hook
kvrp_test_attend_split (no GPU): the stage sequence -- per head group, the
chunks' stages in order -- cut into one contiguous share per block so that each
block moves about the same bytes.  A block pays for the K, V and factor rows of
its stages and, for every segment it holds (a chunk, or the part of it inside
the share), that segment's V_k, query and V_v slots: a share crossing a chunk
boundary takes fewer stages."""
import math

import pytest

SEGMENT_ALLOWANCE = 16384   # bytes a segment is charged beyond its slots (partial, pipeline turn)


@pytest.fixture(scope="module", autouse=True)
def library():
    from position_invariant_kv_gb300.build import build
    build()


def plan(n_q_heads, n_kv_heads, head_dim):
    hg = 4 if n_kv_heads % 4 == 0 else 2 if n_kv_heads % 2 == 0 else 1
    return hg, n_kv_heads // hg, 64 // hg, n_q_heads // n_kv_heads


def costs(tokens, ranks, n_q_heads, n_kv_heads, head_dim, share0):
    """Bytes of each share under the model the split balances."""
    hg, n_hg, ts, g = plan(n_q_heads, n_kv_heads, head_dim)
    nst = [-(-t // ts) for t in tokens]
    segs = []   # (first stage, stages, stage bytes, segment bytes) in sequence order
    f = 0
    for _ in range(n_hg):
        for n, m in zip(nst, ranks):
            sc = ts * (4 * hg * head_dim + 4 * m)
            oc = hg * (2 * head_dim * m + 2 * g * head_dim) + (2 * hg * head_dim * m if m else 0) + SEGMENT_ALLOWANCE
            segs.append((f, n, sc, oc))
            f += n
    out = []
    for a, b in zip(share0, share0[1:]):
        c = 0
        for f0, n, sc, oc in segs:
            lo, hi = max(a, f0), min(b, f0 + n)
            if lo < hi:
                c += (hi - lo) * sc + oc
        out.append(c)
    return out, f


def split(tokens, ranks, n_q_heads, n_kv_heads, head_dim, n_cta):
    import position_invariant_kv_gb300 as kvrp
    return kvrp.kvrp_test_attend_split(tokens, ranks, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads,
                                       head_dim=head_dim, n_cta=n_cta)


def ragged(seed, n, max_tokens, rank_choices):
    import numpy as np
    rng = np.random.default_rng(seed)
    return ([int(x) for x in rng.integers(1, max_tokens + 1, n)],
            [int(rng.choice(rank_choices)) for _ in range(n)])


CASES = {
    # the decode-attention bench: 64 chunks of 4096 tokens, rank 32, 28 / 4 heads x 128
    "bench": ([4096] * 64, [32] * 64, 28, 4, 128, 304),
    # chunks of 17k-23k tokens at mixed ranks: shares of ~16 stages, boundaries inside shares
    "long": ([19000, 23000, 17000, 21000], [16, 32, 0, 16], 8, 4, 64, 304),
    # 200 chunks of 1..90 tokens: many segments per share
    "ragged": ragged(95, 200, 90, [0, 16, 32]) + (8, 2, 128, 304),
    # two head groups of 4 KV heads; one head group of 1 (odd head count)
    "two_groups": ([5000, 3000, 7000], [32, 0, 64], 8, 8, 64, 200),
    "odd_heads": ([8000, 100, 6000], [48, 128, 0], 6, 3, 64, 152),
    # fewer stages than blocks: one stage a share
    "tiny": ([20, 5, 33], [16, 0, 32], 28, 4, 128, 304),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_shares_cover_the_stage_sequence(name):
    tokens, ranks, hq, hkv, d, n_cta = CASES[name]
    share0 = split(tokens, ranks, hq, hkv, d, n_cta)
    _, total = costs(tokens, ranks, hq, hkv, d, [0, 0])
    assert share0[0] == 0 and share0[-1] == total
    assert all(b > a for a, b in zip(share0, share0[1:])), "every share holds a stage"
    assert len(share0) - 1 <= min(n_cta, total)
    if total <= n_cta:
        assert share0 == list(range(total + 1))


@pytest.mark.parametrize("name", ["bench", "long"])
def test_shares_balance_bytes_not_stages(name):
    """Every share but the last costs the same bytes to within the split's granularity:
    about a stage, or half a segment's slots plus a stage where a share stops at a chunk
    boundary rather than pay the next chunk's slots (the last share only ever runs
    short).  A share that crosses a chunk boundary (two segments) holds fewer stages than
    one that does not."""
    tokens, ranks, hq, hkv, d, n_cta = CASES[name]
    share0 = split(tokens, ranks, hq, hkv, d, n_cta)
    c, _ = costs(tokens, ranks, hq, hkv, d, share0)
    hg, n_hg, ts, g = plan(hq, hkv, d)
    stage = max(ts * (4 * hg * d + 4 * m) for m in ranks)
    segment = max(hg * (2 * d * m + 2 * g * d) + (2 * hg * d * m if m else 0) + SEGMENT_ALLOWANCE for m in ranks)
    body = c[:-1]
    assert max(body) - min(body) <= 1.5 * stage + 0.5 * segment, (min(body), max(body), stage, segment)
    assert c[-1] <= max(body)
    if name == "bench":
        hg, n_hg, ts, g = plan(hq, hkv, d)
        per_chunk = -(-4096 // ts)
        sizes = [b - a for a, b in zip(share0, share0[1:])]
        crossing = [i for i, (a, b) in enumerate(zip(share0, share0[1:-1])) if a // per_chunk != (b - 1) // per_chunk]
        whole = [i for i in range(len(sizes) - 1) if i not in crossing]
        assert crossing and whole
        assert max(sizes[i] for i in crossing) < min(sizes[i] for i in whole)


def test_no_tokens_and_bad_arguments():
    assert split([0, 0], [16, 0], 8, 4, 128, 304) == []
    with pytest.raises(ValueError):
        split([100], [16], 8, 3, 128, 304)    # 8 query heads over 3 KV heads
    with pytest.raises(ValueError):
        split([100], [16], 8, 4, 96, 304)     # head_dim 96
    with pytest.raises(ValueError):
        split([100], [16], 8, 4, 128, 0)      # no blocks
    with pytest.raises(ValueError):
        split([100], [16], 34, 2, 128, 304)   # 17 query heads per KV head
