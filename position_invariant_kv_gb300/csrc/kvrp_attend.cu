// Decode attention over relocated, patched chunks, without writing the
// relocated cache (the fused read-side use of the Kamera operator, Kamera,
// gist.science/pt/paper/2606.23581, section 2, "O Operador Kamera").
//
// A chunk is cached in canonical form KV(B|empty) and reused at a new position
// with its shift delta and rank-m patch: K^ = R(delta) K + U_k V_k^T,
// V^ = V + U_v V_v^T.  For one query token the attention over K^, V^ needs
// neither: because R(delta) is orthogonal (a rotation per frequency pair),
//   q . k^_t = (R(-delta) q) . k_t + (V_k,h^T q) . u_k,t,
//   sum_t p_t v^_t = sum_t p_t v_t + V_v,h (sum_t p_t u_v,t),
// so each (chunk, query head) rotates its query once and forms one m-vector
// w = V_k,h^T q; per token the cost is the canonical k_t, v_t and the two rank-m
// rows u_k,t, u_v,t -- the bytes of the canonical cache plus the factors.
//
// Kernels:
//   block_kernel   persistent, two CTAs per SM.  The work is a sequence of
//                  stages -- (head group, chunk, 16 * 4 / hg tokens) -- and each
//                  CTA takes an equal contiguous share of it (stream-K), so
//                  every SM streams the same number of bytes; a chunk, or its
//                  part inside one share, is a segment.  A producer warp fills a
//                  ring of shared-memory slots with bulk copies (the TMA engine):
//                  per segment, first V_k,h and the group's query rows, then the
//                  token stages -- K and V rows (two tokens per copy when one head
//                  group spans the whole row; contiguous rows, or rows of a paged
//                  pool through the chunk's block table) and the U_k, U_v factor
//                  rows, which the group's heads share -- then V_v,h.  Four
//                  consumer warps, one (KV head, 16-token slice) each, turn the
//                  first slots into the rotated, scaled query scale R(-delta) q
//                  (angles in fp64) and w = scale V_k,h^T q, each as a bf16 high
//                  and low part (their sum carries ~16 significant bits); compute
//                  S = K Q^T + U_k W^T with the tokens as the MMA's rows, an online
//                  softmax in registers, and O^T += [V | U_v]^T P^T with P^T
//                  transposed in registers (movmatrix) -- warp-level tensor-core
//                  MMAs (mma.sync m16n8k16 bf16 -> fp32; q, w and P enter as high
//                  + low parts, two products each); and at the segment's end apply
//                  the value patch, O^T += V_v,h (P U_v)^T, from the last slots and
//                  write (O, max, sum) as one fp32 partial.  A consumer never
//                  waits on a global load: everything it reads arrives through
//                  the ring;
//   combine_kernel one CTA per (sequence, query head): merges the partials of
//                  the sequence's chunks in one pass (running max, rescaled
//                  sums), rounds to bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "kvrp.h"
#include "kvrp_plan.h"
#include "kvrp_ptx.h"

namespace kvrp {
namespace attn {

using namespace kvrp::ptx;

constexpr int kMaxChunks = KVRP_ATTN_MAX_CHUNKS;
constexpr int kConsumers = 4;                       // consumer warps; warp kConsumers is the producer
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kSlice = 16;                          // tokens per consumer warp and stage (the MMA's rows)
constexpr int kMaxGroup = 16;                       // query heads per KV head (two n-tiles of 8)
constexpr int kMaxRank = 128;
constexpr int kMaxStages = 8;
constexpr int kCtasPerSm = 2;
constexpr int kMaxCtas = 1024;                      // bound on the block kernel's grid (workspace sizing)
constexpr int kSmemPerSm = 228 * 1024;              // shared memory of one SM, 1 KB of it reserved per CTA

struct ChunkRec {
  const uint16_t *k, *v, *uk, *vk, *uv, *vv;
  const int32_t* table;               // page of each 16 tokens, or null (contiguous rows)
  int32_t n_tokens, rank, seq, st0;   // st0: this chunk's first stage within a head group
  int32_t num_pages;
};

struct Params {
  const uint16_t* q;
  uint16_t* out;
  float* partial;      // [slot][slice][hg * g][d + 2]: O (value patch included), max, sum
  int32_t* seg_cta;    // [2][n_hg][n_chunks]: the first and the last CTA whose share holds
                       // stages of (head group, chunk), written by the block kernel
  uint32_t* status;
  int n_chunks, n_seqs, Hq, Hkv, d, g, m_max;
  int hg;              // KV heads per head group: a power of two dividing Hkv, at most kConsumers
  int n_hg;            // head groups (Hkv / hg)
  int ns;              // token slices per stage (kConsumers / hg)
  int ts;              // tokens per stage (kSlice * ns)
  int stages;          // ring depth
  int row_bytes;       // bytes of one token's head-group row of K (or V): hg * d * 2
  int pair_pitch;      // staged rows go in pairs: token t at (t / 2) * pair_pitch + (t % 2) * row_bytes
  int kv_bytes;        // bytes of a stage's K (and of its V): ts / 2 pairs
  int u_bytes;         // bytes of a stage's U_k (and of its U_v): ts * m_max * 2
  int stage_bytes;
  int hp;              // KV heads per P slot (V_k,h and query rows)
  int hv;              // KV heads per V slot (V_v,h)
  int n_cta;
  int64_t s_hg;        // stages per head group
  float scale;
  double inv_freq[64];   // theta^(-2i/d), i < d/2
  ChunkRec c[kMaxChunks];
  int64_t delta[kMaxChunks];
  int32_t seq_chunk[kMaxChunks + 1];
  int32_t share0[kMaxCtas + 1];   // CTA i takes stages [share0[i], share0[i + 1])
  int32_t n_tok[kMaxChunks];      // tokens of each chunk, packed: the combine reads them lane by lane
};

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t to_bf(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&b);
}
__device__ __forceinline__ uint32_t pack_bf(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

// The query preparation, with every rounding pinned (explicit products and fma, no
// contraction left to the compiler).
//
// (cos, sin) of phi = -delta theta^(-2i/d): phi reduced to [-pi, pi] in fp64 (Cody and
// Waite: 2 pi as a double plus its remainder, each product fused), then sine and
// cosine in fp32.
__device__ __forceinline__ float2 turn_angle(int64_t delta, double inv_freq) {
  const double two_pi_hi = 6.283185307179586, two_pi_lo = 2.4492935982947064e-16;
  const double phi = -static_cast<double>(delta) * inv_freq;
  const double k = rint(phi * (1.0 / 6.283185307179586));
  const double red = fma(-k, two_pi_lo, fma(-k, two_pi_hi, phi));
  float sn, cs;
  sincosf(static_cast<float>(red), &sn, &cs);
  return make_float2(cs, sn);
}
// scale * R(-delta) applied to one frequency pair (a, b) = (q_i, q_{i + d/2}).
__device__ __forceinline__ float2 turn_pair(float a, float b, float2 cs_sn, float scale) {
  return make_float2(__fmul_rn(__fmaf_rn(a, cs_sn.x, -__fmul_rn(b, cs_sn.y)), scale),
                     __fmul_rn(__fmaf_rn(b, cs_sn.x, __fmul_rn(a, cs_sn.y)), scale));
}
// v = high + low, both bf16 (their sum carries ~16 significant bits of v).
__device__ __forceinline__ void split_hl(float v, uint16_t& hi, uint16_t& lo) {
  hi = to_bf(v);
  lo = to_bf(__fsub_rn(v, bf(hi)));
}

// --- the stage sequence ------------------------------------------------------
// Stage f of the whole job is stage (f mod s_hg) of head group f / s_hg; inside a
// head group the chunks follow each other, chunk c owning stages
// [st0, st0 + ceil(n_tokens / ts)).  CTA i takes stages [share0[i], share0[i + 1]),
// boundaries the host places so that every CTA moves about the same bytes.
// The CTA whose share holds stage f: the largest i with share0[i] <= f.
__device__ __forceinline__ int share_of(const Params& p, int64_t f) {
  int lo = 0, hi = p.n_cta - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.share0[mid] <= f) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}
// Position in the stage sequence: head group, chunk, stage within the chunk,
// and the chunk's stage count.  Decoded once per CTA, then advanced.
struct Cursor {
  int hg, c, k, nst;
};
__device__ __forceinline__ Cursor cursor_at(const Params& p, int64_t f) {
  Cursor r;
  r.hg = (int)(f / p.s_hg);
  const int64_t rem = f - (int64_t)r.hg * p.s_hg;
  int lo = 0, hi = p.n_chunks - 1;   // last chunk with st0 <= rem: one with tokens
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.c[mid].st0 <= rem) lo = mid;
    else hi = mid - 1;
  }
  r.c = lo;
  r.k = (int)(rem - p.c[lo].st0);
  r.nst = (p.c[lo].n_tokens + p.ts - 1) / p.ts;
  return r;
}
// The next stage; only called while one exists.
__device__ __forceinline__ void advance(const Params& p, Cursor& r) {
  if (++r.k < r.nst) return;
  r.k = 0;
  do {
    if (++r.c == p.n_chunks) {
      r.c = 0;
      ++r.hg;
    }
  } while (p.c[r.c].n_tokens <= 0);
  r.nst = (p.c[r.c].n_tokens + p.ts - 1) / p.ts;
}
// Partial slot of (CTA i, head group hg, chunk c); distinct for every pair that shares a stage.
__host__ __device__ __forceinline__ int64_t slot_of(int i, int hg, int c, int n_chunks) {
  return (int64_t)i + (int64_t)hg * n_chunks + c;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// The ring slots of one segment (a head group's chunk, or its part inside one CTA's
// share), in order:
//   P slots       V_k,h [d][m] and the query rows [g][d] of p.hp KV heads each (hg / hp
//                 slots): the consumer warps of those heads turn them into the score
//                 product's B fragments;
//   token stages  the K and V rows and the U_k, U_v factor rows of ts tokens;
//   V slots       V_v,h [d][m] of p.hv KV heads each (hg / hv slots; none at rank 0), for
//                 the value patch at the segment's end.
// Everything a consumer reads comes through the ring, issued ahead of its use: under a
// full-bandwidth stream a dependent global load waits microseconds, a ring slot does not.

// From a P slot: this warp's query heads (pairs read from the staged [g][d] rows) and
// V_k,h (staged [d][m]) into the B fragments of the score product -- the rotated, scaled
// query and w = scale V_k,h^T q as high + low bf16 parts, heads >= g zero.  W^T =
// V_k,h^T Q^T on tensor cores (A = V_k,h^T by transposed ldmatrix, B = the raw query
// pairs); angles in fp64, two per lane, handed to the lanes that hold each frequency
// pair by shuffles.  Feature i < d/2 pairs with i + d/2, which sits in k-step
// kk + KT/2 of the same lane, so the rotation is lane-local.
template <int D, int NT, int MCAP>
__device__ __forceinline__ void prepare(const Params& p, uint32_t vks, uint32_t qs, int m, int64_t delta,
                                        uint32_t (&qb)[D / 16][NT][2][2], uint32_t (&wb)[MCAP / 16][NT][2][2]) {
  constexpr int KT = D / 16, RT = MCAP / 16;
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const int t_row = (lane & 7) + ((lane >> 4) << 3), t_col = ((lane >> 3) & 1) * 8;
  const int g = p.g;
  uint32_t raw[KT][NT][2];   // query pairs (head nt 8 + gid; features kk 16 + 2 tig (+ 8) + {0, 1})
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int j = nt * 8 + gid;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      raw[kk][nt][0] = j < g ? lds32(qs + (uint32_t)(j * D + kk * 16 + 2 * tig) * 2) : 0u;
      raw[kk][nt][1] = j < g ? lds32(qs + (uint32_t)(j * D + kk * 16 + 8 + 2 * tig) * 2) : 0u;
    }
  }
  const float2 t0 = turn_angle(delta, p.inv_freq[lane]);   // angles lane and lane + 32
  const float2 t1 = D / 2 > 32 ? turn_angle(delta, p.inv_freq[lane + 32]) : t0;
#pragma unroll
  for (int mt = 0; mt < RT; ++mt) {
    if (mt * 16 >= m) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) wb[mt][nt][0][0] = wb[mt][nt][0][1] = wb[mt][nt][1][0] = wb[mt][nt][1][1] = 0u;
      continue;
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      uint32_t a[4];
      ldsm_x4_trans(a, vks + (uint32_t)((kk * 16 + t_row) * m + mt * 16 + t_col) * 2);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt], a, raw[kk][nt][0], raw[kk][nt][1]);
    }
    // acc = W^T (rank gid (+ 8), heads 2 tig + {0, 1}); its transpose is the B fragment
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      uint16_t h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_hl(__fmul_rn(acc[nt][e], p.scale), h[e], l[e]);
      wb[mt][nt][0][0] = movmatrix_trans(pack_bf(h[0], h[1]));
      wb[mt][nt][0][1] = movmatrix_trans(pack_bf(h[2], h[3]));
      wb[mt][nt][1][0] = movmatrix_trans(pack_bf(l[0], l[1]));
      wb[mt][nt][1][1] = movmatrix_trans(pack_bf(l[2], l[3]));
    }
  }
#pragma unroll
  for (int kk = 0; kk < KT / 2; ++kk) {
    float2 cs[2][2];   // [b0 / b1][element]: angle kk 16 + 8 b + 2 tig + e, held by lane (that) mod 32
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = kk * 16 + 8 * b + 2 * tig + e;
        const float2 t = (kk >> 1) ? t1 : t0;
        cs[b][e] = make_float2(__shfl_sync(0xffffffffu, t.x, i & 31), __shfl_sync(0xffffffffu, t.y, i & 31));
      }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t lo = raw[kk][nt][b], hi = raw[kk + KT / 2][nt][b];
        uint16_t h0[2], l0[2], h1[2], l1[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float2 r = turn_pair(bf((uint16_t)(lo >> (16 * e))), bf((uint16_t)(hi >> (16 * e))), cs[b][e], p.scale);
          split_hl(r.x, h0[e], l0[e]);
          split_hl(r.y, h1[e], l1[e]);
        }
        qb[kk][nt][0][b] = pack_bf(h0[0], h0[1]);
        qb[kk][nt][1][b] = pack_bf(l0[0], l0[1]);
        qb[kk + KT / 2][nt][0][b] = pack_bf(h1[0], h1[1]);
        qb[kk + KT / 2][nt][1][b] = pack_bf(l1[0], l1[1]);
      }
  }
}

// Bounded wait that ignores the abort flag: used to let this CTA's own copies land before it exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint32_t* status) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kTimeoutCycles) {
      if (status) atomicOr(status, KVRP_DEV_TIMEOUT);
      return;
    }
  }
}

template <int D, int NT, int MCAP>   // head dim; n-tiles of 8 query heads; rank the accumulators hold
__global__ void __launch_bounds__(kThreads) block_kernel(const __grid_constant__ Params p) {
  constexpr int KT = D / 16;             // k-steps over the head dim (and m-tiles of the features)
  constexpr int RT = MCAP / 16;          // k-steps over the rank (and m-tiles of the rank columns)
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int64_t f0 = p.share0[cta], f1 = p.share0[cta + 1];
  const uint32_t ring = smem_u32(sm);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kMaxStages + s); };

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kConsumers);
    }
    abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  // the combine kernel may launch (and wait, resident) while this grid runs
  if (tid == 0) pdl_launch_dependents();
  volatile int* abort_p = &abort_flag;
  if (f0 >= f1) return;
  Cursor r = cursor_at(p, f0);

  if (warp == kConsumers) {
    // ---------------- producer ----------------
    // This grid may start while the stream's previous kernel still runs (a programmatic
    // dependent launch): the producer waits for it to complete before its first global
    // access.  Everything the consumers read or write comes after, through the ring.
    pdl_wait();
    const int64_t row = (int64_t)p.Hkv * D;
    const uint32_t row_bytes = (uint32_t)p.row_bytes;
    // one head group covering the whole row: two consecutive tokens (of one page) are one
    // contiguous 2-row source, moved by one copy; otherwise one copy per token row
    const bool pairs = p.n_hg == 1;
    // Page numbers of paged chunks: lane l holds page l % pps of stage batch_f + l / pps
    // (pps pages of 16 tokens per stage), loaded in one batch every 32 / pps stages, so a
    // stage's copies do not wait behind a dependent block-table load of their own.
    const int pps = p.ts / 16;
    const int spb = 32 / pps;
    int64_t batch_f = f1;   // no batch loaded yet
    int32_t pg_lane = 0;
    int s = 0, n_issued = 0;
    uint32_t par = 0;
    // the next slot, once every consumer has released it (the whole warp goes on or stops
    // together: the shuffles below are warp-wide); its shared address, or 0 on an abort
    auto acquire = [&]() -> uint32_t {
      if (!__all_sync(0xffffffffu, wait_phase(empty(s), par ^ 1u, abort_p, p.status))) return 0u;
      return ring + (uint32_t)s * p.stage_bytes;
    };
    auto release = [&]() {
      ++n_issued;
      if (++s == p.stages) {
        s = 0;
        par ^= 1u;
      }
    };
    bool ok = true;
    for (int64_t f = f0; f < f1 && ok;) {
      const ChunkRec& c = p.c[r.c];
      const int m = c.rank;
      const int kv0 = r.hg * p.hg;   // the head group's first KV head
      const int n_tok = (int)min((int64_t)(r.nst - r.k), f1 - f);
      if (lane == 0) {   // for the combine: which CTAs hold this chunk's partials
        const int64_t cell = (int64_t)r.hg * p.n_chunks + r.c;
        if (r.k == 0) p.seg_cta[cell] = cta;
        if (r.k + n_tok == r.nst) p.seg_cta[(int64_t)p.n_hg * p.n_chunks + cell] = cta;
      }
      // P slots
      for (int j = 0; j < p.hg && ok; j += p.hp) {
        const uint32_t st = acquire();
        ok = st != 0u;
        if (!ok) break;
        const uint32_t vk_bytes = (uint32_t)(p.hp * D * m * 2), q_bytes = (uint32_t)(p.hp * p.g * D * 2);
        if (lane == 0) {
          mbar_expect_tx(full(s), vk_bytes + q_bytes);
          if (m > 0) bulk_load(st, c.vk + (int64_t)(kv0 + j) * D * m, vk_bytes, full(s));
          bulk_load(st + vk_bytes, p.q + ((int64_t)c.seq * p.Hq + (int64_t)(kv0 + j) * p.g) * D, q_bytes, full(s));
        }
        release();
      }
      // token stages
      for (int k = 0; k < n_tok && ok; ++k, ++f) {
        const uint32_t st = acquire();
        ok = st != 0u;
        if (!ok) break;
        if (f >= batch_f + spb || batch_f == f1) {
          batch_f = f;
          const int64_t gf = f + lane / pps;
          pg_lane = 0;
          if (gf < f1) {
            const Cursor cl = cursor_at(p, gf);
            const ChunkRec& cc = p.c[cl.c];
            const int pi = cl.k * pps + lane % pps;   // page index within the chunk
            if (cc.table && pi * 16 < cc.n_tokens) pg_lane = __ldg(cc.table + pi);
          }
        }
        const int sbase = (int)(f - batch_f) * pps;
        const int pg_a = __shfl_sync(0xffffffffu, pg_lane, (sbase + (lane >> 4)) & 31);       // token lane
        const int pg_b = __shfl_sync(0xffffffffu, pg_lane, (sbase + 2 + (lane >> 4)) & 31);   // token lane + 32
        const int pg_p = __shfl_sync(0xffffffffu, pg_lane, (sbase + (lane >> 3)) & 31);       // tokens 2 lane, + 1
        const int t0 = r.k * p.ts;
        const int n = min(p.ts, c.n_tokens - t0);
        const uint32_t ub = (uint32_t)n * m * 2;
        if (lane == 0) mbar_expect_tx(full(s), (uint32_t)n * 2 * row_bytes + 2 * ub);
        __syncwarp();
        const int64_t col = (int64_t)kv0 * D;
        // token t of the stage (rows t, t + 1 for a pair; pairs never straddle a page: t0
        // and t are even, pages 16 tokens) lands at (t / 2) pair_pitch
        const int step = pairs ? 2 : 1;
        for (int t = step * lane; t < n; t += 32 * step) {
          int64_t tok = t0 + t;   // the row of this token: contiguous, or page table[tok / 16], slot tok % 16
          if (c.table) {
            int pg = pairs ? pg_p : t < 32 ? pg_a : pg_b;
            if (pg < 0 || pg >= c.num_pages) {
              if (p.status) atomicOr(p.status, KVRP_DEV_BAD_PAGE);
              pg = 0;
            }
            tok = (int64_t)pg * 16 + (tok & 15);
          }
          const uint32_t dst = st + (uint32_t)(t >> 1) * p.pair_pitch + (uint32_t)(t & 1) * row_bytes;
          const uint32_t bytes = (uint32_t)min(step, n - t) * row_bytes;
          bulk_load(dst, c.k + tok * row + col, bytes, full(s));
          bulk_load(dst + p.kv_bytes, c.v + tok * row + col, bytes, full(s));
        }
        if (lane == 0 && ub > 0) {
          bulk_load(st + 2 * p.kv_bytes, c.uk + (int64_t)t0 * m, ub, full(s));
          bulk_load(st + 2 * p.kv_bytes + p.u_bytes, c.uv + (int64_t)t0 * m, ub, full(s));
        }
        release();
        if (f + 1 < f1) advance(p, r);
      }
      // V slots
      if (m > 0)
        for (int j = 0; j < p.hg && ok; j += p.hv) {
          const uint32_t st = acquire();
          ok = st != 0u;
        if (!ok) break;
          const uint32_t vv_bytes = (uint32_t)(p.hv * D * m * 2);
          if (lane == 0) {
            mbar_expect_tx(full(s), vv_bytes);
            bulk_load(st, c.vv + (int64_t)(kv0 + j) * D * m, vv_bytes, full(s));
          }
          release();
        }
    }
    // no copy of this CTA may still be landing when it exits: wait for the last phase issued on each stage
    if (lane == 0)
      for (int j = 0; j < p.stages && j < n_issued; ++j) {
        if (--s < 0) {
          s = p.stages - 1;
          par ^= 1u;
        }
        drain_wait(full(s), par, p.status);
      }
    return;
  }

  // ---------------- consumers: warp -> (KV head hw of the group, token slice sw) ----------------
  const int hw = warp % p.hg, sw = warp / p.hg;
  const int gid = lane >> 2, tig = lane & 3;
  const int g = p.g, pw = D + 2;
  // ldmatrix lane offsets (elements): A from [token][feature] rows; A^T (transposed load) likewise
  const int a_row = lane & 15, a_col = (lane >> 4) * 8;
  const int t_row = (lane & 7) + ((lane >> 4) << 3), t_col = ((lane >> 3) & 1) * 8;
  // this lane's ldmatrix row within a token stage: K rows (A), V rows (A^T, transposed load)
  auto staged = [&](int t) { return (uint32_t)(t >> 1) * p.pair_pitch + (uint32_t)(t & 1) * p.row_bytes; };
  const uint32_t k_lane = staged(sw * kSlice + a_row) + (uint32_t)(hw * D + a_col) * 2;
  const uint32_t v_lane = p.kv_bytes + staged(sw * kSlice + t_row) + (uint32_t)(hw * D + t_col) * 2;

  float o[KT + RT][NT][4];                 // O^T: feature m-tiles, then rank m-tiles (P U_v)
  float mcol[NT][2], lcol[NT][2];
  uint32_t qb[KT][NT][2][2];               // B fragments of Q^T: [k-step][n-tile][high, low][b0, b1]
  uint32_t wb[RT][NT][2][2];               // B fragments of W^T
#pragma unroll
  for (int mt = 0; mt < KT + RT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mcol[nt][0] = mcol[nt][1] = -INFINITY;
    lcol[nt][0] = lcol[nt][1] = 0.f;
  }

  int s = 0;
  uint32_t par = 0;
  auto slot = [&]() { return ring + (uint32_t)s * p.stage_bytes; };
  auto release = [&]() {
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
    if (++s == p.stages) {
      s = 0;
      par ^= 1u;
    }
  };
  bool ok = true;
  for (int64_t f = f0; f < f1 && ok;) {
    const int ci = r.c, hgi = r.hg;
    const ChunkRec& c = p.c[ci];
    const int m = c.rank;
    const int n_tok = (int)min((int64_t)(r.nst - r.k), f1 - f);
    // P slots: this segment's rotated query and w
    for (int j = 0; j < p.hg; j += p.hp) {
      ok = wait_phase(full(s), par, abort_p, p.status);
      if (!ok) break;
      if (hw >= j && hw < j + p.hp)
        prepare<D, NT, MCAP>(p, slot() + (uint32_t)((hw - j) * D * m) * 2,
                             slot() + (uint32_t)(p.hp * D * m + (hw - j) * g * D) * 2, m, p.delta[ci], qb, wb);
      release();
    }
    // token stages
    for (int k = 0; k < n_tok && ok; ++k, ++f) {
      ok = wait_phase(full(s), par, abort_p, p.status);
      if (!ok) break;
      const int nv = min(kSlice, c.n_tokens - (r.k * p.ts + sw * kSlice));   // valid tokens of this slice
      if (nv > 0) {
        const uint32_t st = slot();
        const uint32_t kb = st + k_lane, vb = st + v_lane;
        const uint32_t ukb = st + 2 * p.kv_bytes + (uint32_t)(sw * kSlice * m) * 2;
        const uint32_t uvb = ukb + p.u_bytes;

        // S (16 tokens x 8 NT heads) = K Q^T + U_k W^T, high and low parts in separate chains
        float sh[NT][4], sl[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sh[nt][e] = sl[nt][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
          uint32_t a[4];
          ldsm_x4(a, kb + kk * 32);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(sh[nt], a, qb[kk][nt][0][0], qb[kk][nt][0][1]);
            mma16816(sl[nt], a, qb[kk][nt][1][0], qb[kk][nt][1][1]);
          }
        }
#pragma unroll
        for (int kk = 0; kk < RT; ++kk) {
          if (kk * 16 >= m) break;
          uint32_t a[4];
          ldsm_x4(a, ukb + (uint32_t)(a_row * m + a_col + kk * 16) * 2);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(sh[nt], a, wb[kk][nt][0][0], wb[kk][nt][0][1]);
            mma16816(sl[nt], a, wb[kk][nt][1][0], wb[kk][nt][1][1]);
          }
        }

        // online softmax per head (column): rows are tokens gid (e = 0, 1) and gid + 8 (e = 2, 3)
        float alpha[NT][2];
        uint32_t pb[NT][2][2];   // B fragments of P^T: [n-tile][high, low][tokens 0-7, tokens 8-15]
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float sc[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[e] = sh[nt][e] + sl[nt][e];
          if (gid >= nv) sc[0] = sc[1] = -INFINITY;
          if (gid + 8 >= nv) sc[2] = sc[3] = -INFINITY;
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            float mx = fmaxf(sc[e2], sc[e2 + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(mcol[nt][e2], mx);   // finite: token 0 of the slice is valid
            alpha[nt][e2] = expf(mcol[nt][e2] - mn);     // 0 while nothing was accumulated
            mcol[nt][e2] = mn;
            sc[e2] = expf(sc[e2] - mn);
            sc[e2 + 2] = expf(sc[e2 + 2] - mn);
            lcol[nt][e2] = lcol[nt][e2] * alpha[nt][e2] + (sc[e2] + sc[e2 + 2]);
          }
          uint16_t hb[4], lb[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hb[e] = to_bf(sc[e]);
            lb[e] = to_bf(sc[e] - bf(hb[e]));
          }
          // (token, head) pairs in fragment layout, transposed to (head, token): the B operand
          pb[nt][0][0] = movmatrix_trans(pack_bf(hb[0], hb[1]));
          pb[nt][0][1] = movmatrix_trans(pack_bf(hb[2], hb[3]));
          pb[nt][1][0] = movmatrix_trans(pack_bf(lb[0], lb[1]));
          pb[nt][1][1] = movmatrix_trans(pack_bf(lb[2], lb[3]));
        }

        // O^T = O^T * alpha + [V | U_v]^T P^T: rows features (then rank columns), columns
        // heads.  Past a ragged slice's end the staged rows are whatever a slot last held
        // (never written there this stage): their P is 0 and their V, U_v are masked to 0,
        // so no stale Inf or NaN reaches the sums.
        const uint32_t keep0 = (2 * tig < nv ? 0xffffu : 0u) | (2 * tig + 1 < nv ? 0xffff0000u : 0u);
        const uint32_t keep1 = (8 + 2 * tig < nv ? 0xffffu : 0u) | (9 + 2 * tig < nv ? 0xffff0000u : 0u);
#pragma unroll
        for (int mt = 0; mt < KT + RT; ++mt) {
          if (mt >= KT && (mt - KT) * 16 >= m) break;
          uint32_t a[4];   // A = [V | U_v]^T: a[0], a[1] tokens 2 tig + {0, 1}; a[2], a[3] tokens 8 + 2 tig + {0, 1}
          if (mt < KT) ldsm_x4_trans(a, vb + mt * 32);
          else ldsm_x4_trans(a, uvb + (uint32_t)(t_row * m + t_col + (mt - KT) * 16) * 2);
          if (nv < kSlice) {
            a[0] &= keep0;
            a[1] &= keep0;
            a[2] &= keep1;
            a[3] &= keep1;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            o[mt][nt][0] *= alpha[nt][0];
            o[mt][nt][1] *= alpha[nt][1];
            o[mt][nt][2] *= alpha[nt][0];
            o[mt][nt][3] *= alpha[nt][1];
            mma16816(o[mt][nt], a, pb[nt][0][0], pb[nt][0][1]);
            mma16816(o[mt][nt], a, pb[nt][1][0], pb[nt][1][1]);
          }
        }
      }
      release();
      if (f + 1 < f1) advance(p, r);
    }
    // V slots: the value patch, O^T += V_v,h (P U_v)^T, with the rank rows of O^T as the
    // B operand (fp32 -> high + low bf16, transposed in registers) and the staged V_v,h
    // [d][m] rows as A
    if (m > 0)
      for (int j = 0; j < p.hg && ok; j += p.hv) {
        ok = wait_phase(full(s), par, abort_p, p.status);
      if (!ok) break;
        if (hw >= j && hw < j + p.hv) {
          const uint32_t vvs = slot() + (uint32_t)((hw - j) * D * m) * 2;
#pragma unroll
          for (int rt = 0; rt < RT; ++rt) {
            if (rt * 16 >= m) break;
            uint32_t ub[NT][2][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float* u = o[KT + rt][nt];
              uint16_t hb[4], lb[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                hb[e] = to_bf(u[e]);
                lb[e] = to_bf(u[e] - bf(hb[e]));
              }
              ub[nt][0][0] = movmatrix_trans(pack_bf(hb[0], hb[1]));
              ub[nt][0][1] = movmatrix_trans(pack_bf(hb[2], hb[3]));
              ub[nt][1][0] = movmatrix_trans(pack_bf(lb[0], lb[1]));
              ub[nt][1][1] = movmatrix_trans(pack_bf(lb[2], lb[3]));
            }
#pragma unroll
            for (int ft = 0; ft < KT; ++ft) {
              uint32_t a[4];
              ldsm_x4(a, vvs + (uint32_t)((ft * 16 + a_row) * m + rt * 16 + a_col) * 2);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                mma16816(o[ft][nt], a, ub[nt][0][0], ub[nt][0][1]);
                mma16816(o[ft][nt], a, ub[nt][1][0], ub[nt][1][1]);
              }
            }
          }
        }
        release();
      }
    if (!ok) break;
    // the segment's partial
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        float l = lcol[nt][e2];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        lcol[nt][e2] = l;
      }
    // this warp's partial (its KV head's g query heads) to slot (cta, hg, chunk), slice sw
    float* base = p.partial + ((slot_of(cta, hgi, ci, p.n_chunks) * p.ns + sw) * (p.hg * g) + (int64_t)hw * g) * pw;
#pragma unroll
    for (int ft = 0; ft < KT; ++ft)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = nt * 8 + 2 * tig + (e & 1);
          if (j < g) base[(int64_t)j * pw + ft * 16 + gid + (e >> 1) * 8] = o[ft][nt][e];
        }
    if (gid == 0)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int j = nt * 8 + 2 * tig + e2;
          if (j < g) {
            base[(int64_t)j * pw + D] = mcol[nt][e2];
            base[(int64_t)j * pw + D + 1] = lcol[nt][e2];
          }
        }
#pragma unroll
    for (int mt = 0; mt < KT + RT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mcol[nt][0] = mcol[nt][1] = -INFINITY;
      lcol[nt][0] = lcol[nt][1] = 0.f;
    }
  }
}

// One CTA per (sequence, query head).  Merges the partials of the sequence's
// chunks (a partial with no tokens has max -inf and weight 0) and rounds to bf16.
// The partials of all the sequence's chunks form one list: chunk c contributes one
// entry per token slice for each CTA from the first to the last that holds its stages
// (recorded by the block kernel), so the list is laid out from one round trip to
// memory and a prefix sum in shared memory.  It is then taken in groups of
// kCombineThreads: thread t locates entry t of a group and posts its address; then
// thread -> feature (d = 128) or feature and entry parity (d = 64) loads, for up to
// kBatch entries at once, each entry's max, sum and feature, and folds them into a
// running (max, weighted sum, weighted count): one round trip per kBatch entries.
constexpr int kCombineThreads = 128;
template <int D>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __grid_constant__ Params p) {
  constexpr int G = kCombineThreads / D;   // thread groups, each covering the D features
  constexpr int kBatch = 32;
  __shared__ const float* ent[kCombineThreads];
  __shared__ float part[3][kCombineThreads];
  __shared__ int first_cta[kMaxChunks], prefix[kMaxChunks + 1];
  pdl_wait();   // the block kernel's partials and CTA records
  // the next call's block kernel may start launching: its producer waits for this grid
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int s = blockIdx.x, jq = blockIdx.y, tid = threadIdx.x;
  const int g = p.g, pw = D + 2;
  const int h = jq / g, hg = h / p.hg, row = (h % p.hg) * g + jq % g;
  const int c0 = p.seq_chunk[s], nch = p.seq_chunk[s + 1] - c0;
  // entries of each chunk, then their prefix sum (Hillis and Steele, two values a thread)
  for (int t = tid; t < kMaxChunks; t += kCombineThreads) {
    int n = 0;
    if (t < nch && p.n_tok[c0 + t] > 0) {
      const int64_t cell = (int64_t)hg * p.n_chunks + c0 + t;
      const int i0 = p.seg_cta[cell], i1 = p.seg_cta[(int64_t)p.n_hg * p.n_chunks + cell];
      first_cta[t] = i0;
      n = (i1 - i0 + 1) * p.ns;
    }
    prefix[t + 1] = n;
  }
  if (tid == 0) prefix[0] = 0;
  __syncthreads();
  for (int off = 1; off < kMaxChunks; off <<= 1) {
    int v[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int t = tid + k * kCombineThreads + 1;
      v[k] = t > off ? prefix[t - off] : 0;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 2; ++k) prefix[tid + k * kCombineThreads + 1] += v[k];
    __syncthreads();
  }
  const int n_list = prefix[nch];
  // list entry L: its partial (null past the end)
  auto locate = [&](int L, const float*& pe) {
    pe = nullptr;
    if (L >= n_list) return;
    int lo = 0, hi = nch - 1;   // the chunk: the last k with prefix[k] <= L
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= L) lo = mid;
      else hi = mid - 1;
    }
    const int e = L - prefix[lo];
    pe = p.partial + ((slot_of(first_cta[lo] + e / p.ns, hg, c0 + lo, p.n_chunks) * p.ns + e % p.ns) * (p.hg * g) + row) * pw;
  };
  const int f = tid % D, grp = tid / D;
  float M = -INFINITY, acc = 0.f, den = 0.f;
  for (int L0 = 0; L0 < n_list; L0 += kCombineThreads) {
    const float* pe;
    locate(L0 + tid, pe);
    __syncthreads();   // the previous group's addresses have been read
    ent[tid] = pe;
    __syncthreads();
    const int nx = min(kCombineThreads, n_list - L0);
    for (int x = grp; x < nx; x += kBatch * G) {
      float v[kBatch], mx[kBatch], lt[kBatch];
#pragma unroll
      for (int y = 0; y < kBatch; ++y) {
        const int xy = x + y * G;
        const float* e = xy < nx ? ent[xy] : nullptr;
        mx[y] = e ? e[D] : -INFINITY;
        lt[y] = e ? e[D + 1] : 0.f;
        v[y] = e ? e[f] : 0.f;
      }
      float mb = M;
#pragma unroll
      for (int y = 0; y < kBatch; ++y) mb = fmaxf(mb, mx[y]);
      if (mb == -INFINITY) continue;   // nothing accumulated yet, nothing in this batch
      const float a = expf(M - mb);    // 0 while nothing was accumulated
      acc *= a;
      den *= a;
#pragma unroll
      for (int y = 0; y < kBatch; ++y) {
        const float w = expf(mx[y] - mb);   // 0 for an empty partial
        acc = fmaf(w, v[y], acc);
        den = fmaf(w, lt[y], den);
      }
      M = mb;
    }
  }
  if (G > 1) {   // the groups' running sums, merged by group 0
    part[0][tid] = M;
    part[1][tid] = acc;
    part[2][tid] = den;
    __syncthreads();
    if (grp == 0)
      for (int k = 1; k < G; ++k) {
        const float mk = part[0][k * D + f], mb = fmaxf(M, mk);
        if (mb == -INFINITY) continue;
        const float a = expf(M - mb), b = expf(mk - mb);
        acc = acc * a + part[1][k * D + f] * b;
        den = den * a + part[2][k * D + f] * b;
        M = mb;
      }
  }
  if (grp == 0) p.out[((int64_t)s * p.Hq + jq) * D + f] = to_bf(den > 0.f ? acc / den : 0.f);
}

// ---- host-side planning -----------------------------------------------------
struct Plan {
  int hg, n_hg, ns, ts, row_bytes, pair_pitch, kv_bytes, u_bytes, stage_bytes, stages, hp, hv;
};
Plan make_plan(int n_kv_heads, int head_dim, int m_max, int g) {
  Plan pl;
  pl.hg = 1;
  while (pl.hg * 2 <= kConsumers && n_kv_heads % (pl.hg * 2) == 0) pl.hg *= 2;
  pl.n_hg = n_kv_heads / pl.hg;
  pl.ns = kConsumers / pl.hg;
  pl.ts = kSlice * pl.ns;
  pl.row_bytes = pl.hg * head_dim * 2;
  pl.pair_pitch = 2 * pl.row_bytes + 16;   // +16 bytes a pair: the 8 rows of an ldmatrix phase span 4 bank groups
  pl.kv_bytes = pl.ts / 2 * pl.pair_pitch;
  pl.u_bytes = pl.ts * m_max * 2;
  // a slot holds a token stage, or the P slot (V_k,h and the query rows) or V slot (V_v,h)
  // of at least one KV head; hp, hv: the most KV heads (a power of two) whose P, V slot fits
  const int p_head = head_dim * m_max * 2 + g * head_dim * 2, v_head = head_dim * m_max * 2;
  pl.stage_bytes = (std::max(2 * pl.kv_bytes + 2 * pl.u_bytes, p_head) + 127) / 128 * 128;
  pl.hp = pl.hv = 1;
  while (pl.hp * 2 <= pl.hg && pl.hp * 2 * p_head <= pl.stage_bytes) pl.hp *= 2;
  while (pl.hv * 2 <= pl.hg && pl.hv * 2 * v_head <= pl.stage_bytes) pl.hv *= 2;
  const int budget = kSmemPerSm / kCtasPerSm - 1024 - 256;   // per CTA: reserved and static shared memory
  pl.stages = std::max(2, std::min(kMaxStages, budget / pl.stage_bytes));
  return pl;
}

// Share boundaries over the stage sequence, every CTA's share costing about the same
// bytes: a token stage its K, V and factor rows; every segment a share holds (a chunk,
// or the part of it inside the share) its P and V slots plus kSegmentBytes for the
// partial it writes and the pipeline's turn.  A greedy walk cuts a share once it reaches
// the budget T; bisection finds the smallest T that needs at most n_cta shares.  Writes
// share0[0..count] and returns the count (<= n_cta; every share holds a stage).
constexpr double kSegmentBytes = 16384.0;
int split_shares(const Params& p, int n_cta, int head_dim, int32_t* share0) {
  const int nc = p.n_chunks, D = head_dim;
  std::vector<double> sc(nc), oc(nc);
  std::vector<int> nst(nc);
  double all = 0.0;
  for (int c = 0; c < nc; ++c) {
    const double m = p.c[c].rank;
    nst[c] = (p.c[c].n_tokens + p.ts - 1) / p.ts;
    sc[c] = p.ts * (4.0 * p.hg * D + 4.0 * m);
    oc[c] = p.hg * (2.0 * D * m + 2.0 * p.g * D) + (m > 0 ? 2.0 * p.hg * D * m : 0.0) + kSegmentBytes;
    if (nst[c] > 0) all += p.n_hg * (nst[c] * sc[c] + oc[c]);
  }
  const int64_t total = (int64_t)p.n_hg * p.s_hg;
  auto walk = [&](double T, int32_t* out) {
    int n = 1;
    int64_t f = 0, last = 0;
    double acc = 0.0;
    if (out) out[0] = 0;
    auto cut = [&]() {
      if (out) out[n] = (int32_t)f;
      ++n;
      acc = 0.0;
      last = f;
    };
    for (int hg = 0; hg < p.n_hg; ++hg)
      for (int c = 0; c < nc; ++c) {
        int left = nst[c];
        bool charged = false;
        while (left > 0) {
          if (!charged) {
            // entering the chunk: cut first if that ends this share nearer the budget
            if (f > last && acc + oc[c] + sc[c] - T > T - acc) cut();
            acc += oc[c];
            charged = true;
          }
          int k = left;   // the chunk's remaining stages, or as many as bring the share nearest T
          if (T - acc < k * sc[c]) k = std::max(1, std::min(left, (int)std::floor((T - acc) / sc[c] + 0.5)));
          acc += k * sc[c];
          left -= k;
          f += k;
          if (acc >= T - 0.5 * sc[c] && f < total) {
            cut();
            charged = false;
          }
        }
      }
    if (out) out[n] = (int32_t)total;
    return n;
  };
  double lo = 0.0, hi = all + 1.0;
  for (int it = 0; it < 64 && hi - lo > 1.0; ++it) {
    const double mid = 0.5 * (lo + hi);
    if (walk(mid, nullptr) <= n_cta) hi = mid;
    else lo = mid;
  }
  return walk(hi, share0);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    return kMaxCtas / kCtasPerSm;
  }
  return n;
}

size_t partial_bytes(int n_cta_max, int n_chunks, int Hq, int Hkv, int head_dim) {
  const Plan pl = make_plan(Hkv, head_dim, 0, Hq / Hkv);
  const int64_t slots = n_cta_max + (int64_t)pl.n_hg * n_chunks;
  return sizeof(float) * (size_t)slots * kConsumers * (Hq / Hkv) * (head_dim + 2);
}

}  // namespace attn
}  // namespace kvrp

using namespace kvrp;

extern "C" {

int32_t kvrp_test_attend_split(const int32_t* chunk_tokens, const int32_t* chunk_ranks, int32_t n_chunks,
                               int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t n_cta,
                               int32_t* share0) {
  if (!chunk_tokens || !chunk_ranks || !share0 || n_chunks <= 0 || n_chunks > attn::kMaxChunks || n_kv_heads <= 0 ||
      n_q_heads <= 0 || n_q_heads % n_kv_heads || n_q_heads / n_kv_heads > attn::kMaxGroup ||
      (head_dim != 64 && head_dim != 128) || n_cta <= 0 || n_cta > attn::kMaxCtas)
    return -1;
  int m_max = 0;
  for (int i = 0; i < n_chunks; ++i) {
    if (chunk_tokens[i] < 0 || chunk_ranks[i] < 0 || chunk_ranks[i] > attn::kMaxRank) return -1;
    m_max = std::max(m_max, (int)chunk_ranks[i]);
  }
  const attn::Plan pl = attn::make_plan(n_kv_heads, head_dim, m_max, n_q_heads / n_kv_heads);
  std::vector<uint8_t> mem(sizeof(attn::Params), 0);   // ~29 KB: off the stack
  attn::Params& p = *reinterpret_cast<attn::Params*>(mem.data());
  p.n_chunks = n_chunks;
  p.g = n_q_heads / n_kv_heads;
  p.hg = pl.hg;
  p.n_hg = pl.n_hg;
  p.ts = pl.ts;
  int64_t st0 = 0;
  for (int i = 0; i < n_chunks; ++i) {
    p.c[i].n_tokens = chunk_tokens[i];
    p.c[i].rank = chunk_ranks[i];
    p.c[i].st0 = (int32_t)st0;
    st0 += (chunk_tokens[i] + pl.ts - 1) / pl.ts;
  }
  p.s_hg = st0;
  const int64_t total = (int64_t)p.n_hg * p.s_hg;
  if (total == 0) return 0;
  if (total > INT32_MAX) return -1;
  return attn::split_shares(p, (int)std::min<int64_t>(n_cta, total), head_dim, share0);
}

size_t kv_attend_relocated_workspace_size(int32_t n_chunks, const int32_t* chunk_tokens, int32_t n_q_heads,
                                          int32_t n_kv_heads, int32_t head_dim) {
  if (n_chunks <= 0 || !chunk_tokens || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads || head_dim <= 0)
    return 0;
  const int n_cta_max = std::min(attn::kMaxCtas, attn::kCtasPerSm * attn::sm_count());
  const size_t part = (attn::partial_bytes(n_cta_max, n_chunks, n_q_heads, n_kv_heads, head_dim) + 255) / 256 * 256;
  return part + 2 * sizeof(int32_t) * (size_t)n_kv_heads * n_chunks + 256;
}

kvrp_status kv_attend_relocated(const void* q, const kvrp_attn_chunk* chunks, int32_t n_chunks,
                                const int32_t* seq_chunks, int32_t n_seqs, int32_t n_q_heads, int32_t n_kv_heads,
                                int32_t head_dim, double rope_theta, float softmax_scale, void* out,
                                void* workspace, size_t workspace_bytes, uint32_t* d_status, kvrp_stream_t stream) {
  g_last_launches = 0;
  if (!q || !chunks || !seq_chunks || !out) return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: NULL argument");
  if (n_chunks <= 0 || n_chunks > attn::kMaxChunks)
    return fail(KVRP_ERR_UNSUPPORTED, "kv_attend_relocated: 1 <= n_chunks <= %d", attn::kMaxChunks);
  if (n_seqs <= 0 || n_seqs > 65535) return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: 1 <= n_seqs <= 65535");
  if (head_dim != 64 && head_dim != 128)
    return fail(KVRP_ERR_UNSUPPORTED, "kv_attend_relocated: head_dim must be 64 or 128");
  if (n_kv_heads <= 0 || n_q_heads <= 0 || n_q_heads % n_kv_heads || n_q_heads / n_kv_heads > attn::kMaxGroup)
    return fail(KVRP_ERR_UNSUPPORTED, "kv_attend_relocated: n_q_heads must be a multiple of n_kv_heads, at most %d x",
                attn::kMaxGroup);
  if (!(rope_theta > 0.0) || !std::isfinite(rope_theta) || !(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: rope_theta and softmax_scale must be > 0");
  if (!aligned16(q) || !aligned16(out)) return fail(KVRP_ERR_ALIGNMENT, "kv_attend_relocated: q, out not 16-byte aligned");
  if (seq_chunks[0] != 0 || seq_chunks[n_seqs] != n_chunks)
    return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: seq_chunks must run from 0 to n_chunks");
  for (int s = 0; s < n_seqs; ++s)
    if (seq_chunks[s + 1] < seq_chunks[s])
      return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: seq_chunks must not decrease");
  std::vector<int32_t> tok(n_chunks);
  int m_max = 0;
  int64_t all_tokens = 0;
  for (int i = 0; i < n_chunks; ++i) {
    const kvrp_attn_chunk& c = chunks[i];
    if (c.n_tokens < 0) return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: chunk %d: n_tokens < 0", i);
    if (c.n_tokens > 0 && (!c.k || !c.v)) return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: chunk %d: NULL k/v", i);
    if (c.rank < 0 || c.rank > attn::kMaxRank || c.rank % 16)
      return fail(KVRP_ERR_UNSUPPORTED, "kv_attend_relocated: chunk %d: rank must be 0 or a multiple of 16 up to %d", i,
                  attn::kMaxRank);
    if (c.rank > 0 && (!c.uk || !c.vk || !c.uv || !c.vv))
      return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: chunk %d: rank > 0 needs all four factors", i);
    if ((c.k && !aligned16(c.k)) || (c.v && !aligned16(c.v)) || (c.uk && !aligned16(c.uk)) || (c.uv && !aligned16(c.uv)) ||
        (c.vk && !aligned16(c.vk)) || (c.vv && !aligned16(c.vv)))
      return fail(KVRP_ERR_ALIGNMENT, "kv_attend_relocated: chunk %d: pointers must be 16-byte aligned", i);
    if (c.block_table && c.num_pages <= 0)
      return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: chunk %d: a block table needs num_pages > 0", i);
    if (c.block_table && reinterpret_cast<uintptr_t>(c.block_table) % 4)
      return fail(KVRP_ERR_ALIGNMENT, "kv_attend_relocated: chunk %d: block table not 4-byte aligned", i);
    tok[i] = c.n_tokens;
    m_max = std::max(m_max, (int)c.rank);
    all_tokens += c.n_tokens;
  }
  if (all_tokens > INT32_MAX)
    return fail(KVRP_ERR_UNSUPPORTED, "kv_attend_relocated: at most 2^31 - 1 tokens per call");
  const size_t need = kv_attend_relocated_workspace_size(n_chunks, tok.data(), n_q_heads, n_kv_heads, head_dim);
  if (!workspace || workspace_bytes < need)
    return fail(KVRP_ERR_WORKSPACE, "kv_attend_relocated: workspace of %zu bytes needed", need);

  const attn::Plan pl = attn::make_plan(n_kv_heads, head_dim, m_max, n_q_heads / n_kv_heads);
  static_assert(sizeof(attn::Params) <= 32000, "kernel parameter block too large");
  attn::Params* pp = new attn::Params;   // ~20 KB: off the stack
  std::memset(pp, 0, sizeof(attn::Params));
  attn::Params& p = *pp;
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  p.status = d_status;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255));
  p.partial = reinterpret_cast<float*>(base);
  {
    const int n_cta_max = std::min(attn::kMaxCtas, attn::kCtasPerSm * attn::sm_count());
    const size_t part = (attn::partial_bytes(n_cta_max, n_chunks, n_q_heads, n_kv_heads, head_dim) + 255) / 256 * 256;
    p.seg_cta = reinterpret_cast<int32_t*>(base + part);
  }
  p.n_chunks = n_chunks;
  p.n_seqs = n_seqs;
  p.Hq = n_q_heads;
  p.Hkv = n_kv_heads;
  p.d = head_dim;
  p.g = n_q_heads / n_kv_heads;
  p.m_max = m_max;
  p.hg = pl.hg;
  p.n_hg = pl.n_hg;
  p.ns = pl.ns;
  p.ts = pl.ts;
  p.stages = pl.stages;
  p.row_bytes = pl.row_bytes;
  p.pair_pitch = pl.pair_pitch;
  p.kv_bytes = pl.kv_bytes;
  p.u_bytes = pl.u_bytes;
  p.stage_bytes = pl.stage_bytes;
  p.hp = pl.hp;
  p.hv = pl.hv;
  p.scale = softmax_scale;
  for (int i = 0; i < head_dim / 2; ++i) p.inv_freq[i] = std::pow(rope_theta, -2.0 * i / head_dim);
  int64_t st0 = 0;
  for (int s = 0; s < n_seqs; ++s)
    for (int i = seq_chunks[s]; i < seq_chunks[s + 1]; ++i) {
      const kvrp_attn_chunk& c = chunks[i];
      attn::ChunkRec& r = p.c[i];
      r.k = static_cast<const uint16_t*>(c.k);
      r.v = static_cast<const uint16_t*>(c.v);
      r.uk = static_cast<const uint16_t*>(c.uk);
      r.vk = static_cast<const uint16_t*>(c.vk);
      r.uv = static_cast<const uint16_t*>(c.uv);
      r.vv = static_cast<const uint16_t*>(c.vv);
      r.table = c.block_table;
      r.num_pages = c.block_table ? c.num_pages : 0;
      r.n_tokens = c.n_tokens;
      p.n_tok[i] = c.n_tokens;
      r.rank = c.rank;
      r.seq = s;
      r.st0 = (int32_t)st0;
      p.delta[i] = c.delta;
      st0 += (c.n_tokens + pl.ts - 1) / pl.ts;
    }
  p.s_hg = st0;
  if ((int64_t)p.n_hg * p.s_hg > INT32_MAX) {
    delete pp;
    return fail(KVRP_ERR_UNSUPPORTED, "kv_attend_relocated: at most 2^31 - 1 stages per call");
  }
  for (int s = 0; s <= n_seqs; ++s) p.seq_chunk[s] = seq_chunks[s];

  cudaStream_t st = stream;
  void (*blk_fn)(attn::Params) = nullptr;
  const bool two = p.g > 8, big = m_max > 32;
  if (head_dim == 64)
    blk_fn = two ? (big ? attn::block_kernel<64, 2, 128> : attn::block_kernel<64, 2, 32>)
                 : (big ? attn::block_kernel<64, 1, 128> : attn::block_kernel<64, 1, 32>);
  else
    blk_fn = two ? (big ? attn::block_kernel<128, 2, 128> : attn::block_kernel<128, 2, 32>)
                 : (big ? attn::block_kernel<128, 1, 128> : attn::block_kernel<128, 1, 32>);
  const int smem = pl.stages * pl.stage_bytes;
  cudaError_t e = cudaFuncSetAttribute(blk_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  int per_sm = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, blk_fn, attn::kThreads, smem);
  const int n_cta_max = std::min(attn::kMaxCtas, attn::kCtasPerSm * attn::sm_count());
  p.n_cta = (int)std::max<int64_t>(1, std::min<int64_t>({(int64_t)std::max(per_sm, 1) * attn::sm_count(), (int64_t)n_cta_max,
                                                         (int64_t)p.n_hg * p.s_hg}));
  if (p.s_hg > 0) p.n_cta = attn::split_shares(p, p.n_cta, head_dim, p.share0);
  // Both kernels are programmatic dependent launches: each may start while the kernel
  // before it on the stream runs, and waits (griddepcontrol.wait) for that kernel to
  // complete before it touches global memory -- the block kernel in its producer, the
  // combine before it reads the partials.
  int launches = 0;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cfg.attrs = attr;
  if (e == cudaSuccess && p.s_hg > 0) {
    cfg.gridDim = dim3(p.n_cta);
    cfg.blockDim = dim3(attn::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.numAttrs = 1;   // its producer waits (griddepcontrol.wait) before any global access
    e = cudaLaunchKernelEx(&cfg, blk_fn, p);
    ++launches;
  }
  if (e == cudaSuccess) {
    cfg.gridDim = dim3(n_seqs, n_q_heads);
    cfg.blockDim = dim3(attn::kCombineThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, head_dim == 64 ? attn::combine_kernel<64> : attn::combine_kernel<128>, p);
    ++launches;
  }
  g_last_launches = e == cudaSuccess ? launches : 0;
  delete pp;
  if (e != cudaSuccess) return fail(KVRP_ERR_CUDA, "kv_attend_relocated: %s", cudaGetErrorString(e));
  return KVRP_OK;
}

}  // extern "C"
