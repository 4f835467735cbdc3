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
//   prep_kernel    one CTA per (chunk, KV head): the rotated, scaled queries
//                  scale * R(-delta) q (angles in fp64) and w = scale V_k,h^T q
//                  of the group's query heads, each split into a bf16 high and
//                  low part (their sum carries ~16 significant bits);
//   block_kernel   one CTA per (block of up to 256 tokens of one chunk, KV
//                  head), four warps; 64-token sub-blocks stream through a
//                  double-buffered cp.async pipeline (one barrier each) and
//                  every warp owns 16 tokens of each: S^T = Q K^T + W U_k^T
//                  (query heads as the 16 rows), an online softmax in
//                  registers, and O += P [V | U_v] with P taken straight from
//                  the score accumulators -- all products warp-level
//                  tensor-core MMAs (mma.sync m16n8k16 bf16 -> fp32, fragments
//                  by ldmatrix; q, w and P enter as high + low bf16 parts,
//                  two products each).  The four warps' (O, max, sum) merge in
//                  shared memory into one fp32 partial per block and head;
//   combine_kernel one CTA per (sequence, query head): merges the partials of
//                  the sequence's blocks by their maxima, applies each chunk's
//                  value patch V_v,h (P U_v) once, rounds to bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "kvrp.h"
#include "kvrp_plan.h"

namespace kvrp {
namespace at {

constexpr int kMaxChunks = KVRP_ATTN_MAX_CHUNKS;
constexpr int kBlock = 64;          // tokens per sub-block
constexpr int kSubs = 4;            // sub-blocks per block_kernel CTA
constexpr int kCta = kBlock * kSubs;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxGroup = 16;       // query heads per KV head (one m16 tile)
constexpr int kMaxRank = 128;

struct ChunkRec {
  const uint16_t *k, *v, *uk, *vk, *uv, *vv;
  int32_t n_tokens, rank, seq, blk0;   // blk0: first block of this chunk
};

struct Params {
  const uint16_t* q;
  uint16_t* out;
  float* partial;      // [n_blocks][Hq][d + m_max + 2]: P V, P U_v, max, sum
  uint16_t* qhl;       // [n_chunks][2][Hq][d]: high, low bf16 parts of scale * R(-delta) q
  uint16_t* whl;       // [n_chunks][2][Hq][m_max]: high, low parts of scale * V_k,h^T q
  int n_chunks, n_seqs, n_blocks, Hq, Hkv, d, g, m_max;
  float scale;
  double theta;
  ChunkRec c[kMaxChunks];
  int64_t delta[kMaxChunks];
  int32_t seq_chunk[kMaxChunks + 1];
};

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t to_bf(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&b);
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__global__ void __launch_bounds__(256) prep_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint16_t vks[];   // V_k,h [d][m]
  __shared__ float2 rot[64];                         // (cos, sin) of -delta * theta^(-2i/d)
  const int ci = blockIdx.x, h = blockIdx.y;
  const ChunkRec& c = p.c[ci];
  const int d = p.d, half = d / 2, g = p.g, m = c.rank, Hq = p.Hq;
  const uint16_t* q = p.q + ((int64_t)c.seq * Hq + (int64_t)h * g) * d;
  uint16_t* qh = p.qhl + ((int64_t)ci * 2 * Hq + (int64_t)h * g) * d;
  uint16_t* ql = qh + (int64_t)Hq * d;
  if (m > 0)
    for (int e = threadIdx.x; e < d * m / 8; e += blockDim.x)
      reinterpret_cast<uint4*>(vks)[e] = reinterpret_cast<const uint4*>(c.vk + (int64_t)h * d * m)[e];
  if (threadIdx.x < half) {
    const int i = threadIdx.x;
    const double phi = -static_cast<double>(p.delta[ci]) * pow(p.theta, -2.0 * i / d);
    rot[i] = make_float2((float)cos(phi), (float)sin(phi));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < g * half; e += blockDim.x) {
    const int j = e / half, i = e - j * half;
    const float cs = rot[i].x, sn = rot[i].y;
    const float a = bf(q[j * d + i]), b = bf(q[j * d + i + half]);
    const float r0 = (a * cs - b * sn) * p.scale, r1 = (b * cs + a * sn) * p.scale;
    const uint16_t h0 = to_bf(r0), h1 = to_bf(r1);
    qh[j * d + i] = h0;
    qh[j * d + i + half] = h1;
    ql[j * d + i] = to_bf(r0 - bf(h0));
    ql[j * d + i + half] = to_bf(r1 - bf(h1));
  }
  if (m == 0) return;
  uint16_t* wh = p.whl + ((int64_t)ci * 2 * Hq + (int64_t)h * g) * p.m_max;
  uint16_t* wl = wh + (int64_t)Hq * p.m_max;
  for (int e = threadIdx.x; e < g * m; e += blockDim.x) {
    const int j = e / m, r = e - j * m;
    float a4[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < d; i += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) a4[u] = fmaf(bf(vks[(i + u) * m + r]), bf(q[j * d + i + u]), a4[u]);
    }
    const float w = ((a4[0] + a4[1]) + (a4[2] + a4[3])) * p.scale;
    const uint16_t hw = to_bf(w);
    wh[j * p.m_max + r] = hw;
    wl[j * p.m_max + r] = to_bf(w - bf(hw));
  }
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Warp-level tensor-core product D += A B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// A fragment (16 x 16, row-major source): lane l addresses row (l & 15), column 8 (l >> 4)
__device__ __forceinline__ void ldsm_a(uint32_t (&r)[4], const uint16_t* base, int pitch) {
  const int l = threadIdx.x & 31;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(base + (l & 15) * pitch + (l >> 4) * 8)));
}
// B fragment (16 x 8) from an [n][k] row-major source: lane l < 16 addresses row (l & 7), column 8 (l >> 3)
__device__ __forceinline__ void ldsm_b(uint32_t (&r)[2], const uint16_t* base, int pitch) {
  const int l = threadIdx.x & 15;
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(base + (l & 7) * pitch + (l >> 3) * 8)));
}
// B fragment (16 x 8) from a [k][n] row-major source (transposed load): lane l < 16 addresses row l
__device__ __forceinline__ void ldsm_bt(uint32_t (&r)[2], const uint16_t* base, int pitch) {
  const int l = threadIdx.x & 15;
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(base + l * pitch)));
}

// Two B fragments (16 x 8 each, n-tiles n0 and n0 + 8) from an [n][k] row-major source
__device__ __forceinline__ void ldsm_b2(uint32_t (&r)[4], const uint16_t* base, int pitch) {
  const int l = threadIdx.x & 31;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(base + ((l & 7) + ((l >> 4) << 3)) * pitch + ((l >> 3) & 1) * 8)));
}
// Two B fragments (n-tiles n0 and n0 + 8) from a [k][n] row-major source (transposed load)
__device__ __forceinline__ void ldsm_bt2(uint32_t (&r)[4], const uint16_t* base, int pitch) {
  const int l = threadIdx.x & 31;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(base + (l & 15) * pitch + (l >> 4) * 8)));
}
__device__ __forceinline__ uint32_t pack_bf(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

// Shared memory of block_kernel (bf16 rows padded by 16 bytes for conflict-free ldmatrix).
struct BlockSmem {
  int kv_pitch, u_pitch, m_pitch;
  int k_off, v_off, uk_off, uv_off, buf_bytes;   // buffer b of a stage at (offset + b * buf_bytes)
  int qh_off, ql_off, wh_off, wl_off;
  int bytes;
};
// Staging (two buffers of K, V, U_k, U_v), then the queries and w; the warps'
// final (O, max, sum) reuse the staging area (fp32 rows of m_pitch floats).
__host__ __device__ inline BlockSmem block_smem(int d, int m) {
  BlockSmem s;
  s.kv_pitch = d + 8;
  s.u_pitch = (m > 0 ? m : 16) + 8;
  s.m_pitch = d + m + 8;
  int off = 0;
  s.k_off = off; off += kBlock * s.kv_pitch * 2;
  s.v_off = off; off += kBlock * s.kv_pitch * 2;
  s.uk_off = off; off += m > 0 ? kBlock * s.u_pitch * 2 : 0;
  s.uv_off = off; off += m > 0 ? kBlock * s.u_pitch * 2 : 0;
  s.buf_bytes = off;
  off *= 2;
  const int merge = kWarps * kMaxGroup * (s.m_pitch + 2) * 4;
  off = off > merge ? off : merge;
  s.qh_off = off; off += kMaxGroup * s.kv_pitch * 2;
  s.ql_off = off; off += kMaxGroup * s.kv_pitch * 2;
  s.wh_off = off; off += m > 0 ? kMaxGroup * s.u_pitch * 2 : 0;
  s.wl_off = off; off += m > 0 ? kMaxGroup * s.u_pitch * 2 : 0;
  s.bytes = off;
  return s;
}

__device__ __forceinline__ int chunk_of_block(const Params& p, int blk) {
  int lo = 0, hi = p.n_chunks - 1;   // last chunk whose blk0 <= blk
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (p.c[mid].blk0 <= blk) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int D, int UT>   // head dim; rank n-tiles the accumulators hold (rank <= 8 UT)
__global__ void __launch_bounds__(kThreads) block_kernel(const __grid_constant__ Params p) {
  constexpr int DT = D / 8, CPR = D / 8;
  extern __shared__ __align__(16) uint8_t sm[];
  const int blk = blockIdx.x, h = blockIdx.y;
  const int ci = chunk_of_block(p, blk);
  const ChunkRec& c = p.c[ci];
  const int t0 = (blk - c.blk0) * kCta;
  const int n_sub = (min(kCta, c.n_tokens - t0) + kBlock - 1) / kBlock;
  const int g = p.g, m = c.rank, row = p.Hkv * D, upr = m / 8, ntu = m / 8;
  const BlockSmem L = block_smem(D, p.m_max);
  uint16_t* qhs = reinterpret_cast<uint16_t*>(sm + L.qh_off);
  uint16_t* qls = reinterpret_cast<uint16_t*>(sm + L.ql_off);
  uint16_t* whs = reinterpret_cast<uint16_t*>(sm + L.wh_off);
  uint16_t* wls = reinterpret_cast<uint16_t*>(sm + L.wl_off);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;

  // one sub-block (64 tokens from token ts) into buffer b; rows past the chunk end are zero
  auto stage = [&](int b, int ts) {
    const int n = min(kBlock, c.n_tokens - ts);
    uint16_t* ks = reinterpret_cast<uint16_t*>(sm + L.k_off + b * L.buf_bytes);
    uint16_t* vs = reinterpret_cast<uint16_t*>(sm + L.v_off + b * L.buf_bytes);
#pragma unroll
    for (int e = tid; e < kBlock * CPR; e += kThreads) {
      const int r = e / CPR, q16 = e % CPR;
      const bool ok = r < n;
      const int64_t off = (int64_t)(ts + r) * row + h * D + 8 * q16;
      cp_async16(ks + r * L.kv_pitch + 8 * q16, ok ? c.k + off : c.k, ok);
      cp_async16(vs + r * L.kv_pitch + 8 * q16, ok ? c.v + off : c.v, ok);
    }
    if (m > 0) {
      uint16_t* uks = reinterpret_cast<uint16_t*>(sm + L.uk_off + b * L.buf_bytes);
      uint16_t* uvs = reinterpret_cast<uint16_t*>(sm + L.uv_off + b * L.buf_bytes);
      for (int e = tid; e < kBlock * upr; e += kThreads) {
        const int r = e / upr, q16 = e - r * upr;
        const bool ok = r < n;
        const int64_t off = (int64_t)(ts + r) * m + 8 * q16;
        cp_async16(uks + r * L.u_pitch + 8 * q16, ok ? c.uk + off : c.uk, ok);
        cp_async16(uvs + r * L.u_pitch + 8 * q16, ok ? c.uv + off : c.uv, ok);
      }
    }
    cp_async_commit();
  };

  // the queries and w of this head group (rows g..15 zero), then the first sub-block
  const uint16_t* qsrc = p.qhl + ((int64_t)ci * 2 * p.Hq + (int64_t)h * g) * D;
  for (int e = tid; e < 2 * kMaxGroup * CPR; e += kThreads) {
    const int part = e / (kMaxGroup * CPR), rr = e % (kMaxGroup * CPR);
    const int j = rr / CPR, q16 = rr % CPR;
    const bool ok = j < g;
    cp_async16((part ? qls : qhs) + j * L.kv_pitch + 8 * q16,
               ok ? qsrc + (int64_t)part * p.Hq * D + (int64_t)j * D + 8 * q16 : qsrc, ok);
  }
  if (m > 0) {
    const uint16_t* wsrc = p.whl + ((int64_t)ci * 2 * p.Hq + (int64_t)h * g) * p.m_max;
    for (int e = tid; e < 2 * kMaxGroup * upr; e += kThreads) {
      const int part = e / (kMaxGroup * upr), rr = e - part * kMaxGroup * upr;
      const int j = rr / upr, q16 = rr - j * upr;
      const bool ok = j < g;
      cp_async16((part ? wls : whs) + j * L.u_pitch + 8 * q16,
                 ok ? wsrc + (int64_t)part * p.Hq * p.m_max + (int64_t)j * p.m_max + 8 * q16 : wsrc, ok);
    }
  }
  stage(0, t0);

  // this warp's running state: rows gid and gid + 8 (query heads) of O = [P V | P U_v]
  float o[DT + UT][4] = {};
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int tok0 = warp * 16;   // this warp's 16 tokens of each sub-block

  for (int sb = 0; sb < n_sub; ++sb) {
    const int b = sb & 1;
    const int ts = t0 + sb * kBlock;
    const int n = min(kBlock, c.n_tokens - ts);
    cp_async_wait<0>();
    __syncthreads();   // sub-block sb is visible; every warp is done with buffer b ^ 1
    if (sb + 1 < n_sub) stage(b ^ 1, ts + kBlock);
    if (tok0 >= n) continue;   // warp-uniform: this slice lies past the chunk end
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(sm + L.k_off + b * L.buf_bytes) + tok0 * L.kv_pitch;
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(sm + L.v_off + b * L.buf_bytes) + tok0 * L.kv_pitch;
    const uint16_t* uks = reinterpret_cast<const uint16_t*>(sm + L.uk_off + b * L.buf_bytes) + tok0 * L.u_pitch;
    const uint16_t* uvs = reinterpret_cast<const uint16_t*>(sm + L.uv_off + b * L.buf_bytes) + tok0 * L.u_pitch;

    // S^T (16 heads x 16 tokens, two n-tiles) = Q K^T + W U_k^T
    float s[2][4] = {};
#pragma unroll
    for (int k0 = 0; k0 < D; k0 += 16) {
      uint32_t ah[4], al[4], bk[4];
      ldsm_a(ah, qhs + k0, L.kv_pitch);
      ldsm_a(al, qls + k0, L.kv_pitch);
      ldsm_b2(bk, ks + k0, L.kv_pitch);
      const uint32_t b0[2] = {bk[0], bk[1]}, b1[2] = {bk[2], bk[3]};
      mma16816(s[0], ah, b0);
      mma16816(s[1], ah, b1);
      mma16816(s[0], al, b0);
      mma16816(s[1], al, b1);
    }
    for (int k0 = 0; k0 < m; k0 += 16) {
      uint32_t ah[4], al[4], bk[4];
      ldsm_a(ah, whs + k0, L.u_pitch);
      ldsm_a(al, wls + k0, L.u_pitch);
      ldsm_b2(bk, uks + k0, L.u_pitch);
      const uint32_t b0[2] = {bk[0], bk[1]}, b1[2] = {bk[2], bk[3]};
      mma16816(s[0], ah, b0);
      mma16816(s[1], ah, b1);
      mma16816(s[0], al, b0);
      mma16816(s[1], al, b1);
    }

    // online softmax over this warp's tokens: row r of the fragment is head gid + 8 r
    float alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = tok0 + nt * 8 + 2 * tig + e;
          if (t >= n) s[nt][2 * r + e] = -INFINITY;
          mx = fmaxf(mx, s[nt][2 * r + e]);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(mrow[r], mx);   // finite: token tok0 < n is in every quad's row
      alpha[r] = expf(mrow[r] - m_new);         // 0 while nothing was accumulated
      mrow[r] = m_new;
      float sum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float pe = expf(s[nt][2 * r + e] - m_new);
          s[nt][2 * r + e] = pe;
          sum += pe;
        }
      lrow[r] = lrow[r] * alpha[r] + sum;
    }
    // P (16 heads x 16 tokens) as the A operand, high and low bf16 parts
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float p0 = s[x >> 1][2 * (x & 1)], p1 = s[x >> 1][2 * (x & 1) + 1];
      const uint16_t h0 = to_bf(p0), h1 = to_bf(p1);
      ph[x] = pack_bf(h0, h1);
      pl[x] = pack_bf(to_bf(p0 - bf(h0)), to_bf(p1 - bf(h1)));
    }

    // O = O * alpha + P [V | U_v], two n-tiles per transposed load
#pragma unroll
    for (int x = 0; x < DT + UT; x += 2) {
      if (x >= DT && x - DT >= ntu) break;
      uint32_t bv[4];
      if (x < DT) ldsm_bt2(bv, vs + x * 8, L.kv_pitch);
      else ldsm_bt2(bv, uvs + (x - DT) * 8, L.u_pitch);
      const uint32_t b0[2] = {bv[0], bv[1]}, b1[2] = {bv[2], bv[3]};
#pragma unroll
      for (int y = 0; y < 2; ++y) {
        o[x + y][0] *= alpha[0]; o[x + y][1] *= alpha[0];
        o[x + y][2] *= alpha[1]; o[x + y][3] *= alpha[1];
      }
      mma16816(o[x], ph, b0);
      mma16816(o[x + 1], ph, b1);
      mma16816(o[x], pl, b0);
      mma16816(o[x + 1], pl, b1);
    }
  }

  // merge the four warps: each writes (O, max, sum) of its rows; then one pass over (head, column)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
  }
  __syncthreads();   // every warp is done with the staging buffers (no copy is in flight)
  float* mo = reinterpret_cast<float*>(sm);                       // [warp][16][m_pitch]
  float* ml = mo + kWarps * kMaxGroup * L.m_pitch;                // [warp][16][2]: max, sum
  {
    float* mw = mo + warp * kMaxGroup * L.m_pitch;
#pragma unroll
    for (int x = 0; x < DT + UT; ++x) {
      if (x >= DT && x - DT >= ntu) break;
      const int col = (x < DT ? x * 8 : D + (x - DT) * 8) + 2 * tig;
      *reinterpret_cast<float2*>(mw + gid * L.m_pitch + col) = make_float2(o[x][0], o[x][1]);
      *reinterpret_cast<float2*>(mw + (gid + 8) * L.m_pitch + col) = make_float2(o[x][2], o[x][3]);
    }
    if (tig == 0) {
      ml[(warp * kMaxGroup + gid) * 2] = mrow[0];
      ml[(warp * kMaxGroup + gid) * 2 + 1] = lrow[0];
      ml[(warp * kMaxGroup + gid + 8) * 2] = mrow[1];
      ml[(warp * kMaxGroup + gid + 8) * 2 + 1] = lrow[1];
    }
  }
  __syncthreads();
  const int pw = D + p.m_max + 2, cols = D + m;
  float* part = p.partial + ((int64_t)blk * p.Hq + (int64_t)h * g) * pw;
  for (int e = tid; e < g * (cols + 2); e += kThreads) {
    const int j = e / (cols + 2), col = e - j * (cols + 2);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml[(w * kMaxGroup + j) * 2]);
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = ml[(w * kMaxGroup + j) * 2];
      const float sc = mw == -INFINITY ? 0.f : expf(mw - M);
      const float v = col < cols ? mo[(w * kMaxGroup + j) * L.m_pitch + col]
                                 : (col == cols ? 0.f : ml[(w * kMaxGroup + j) * 2 + 1]);
      acc = fmaf(sc, v, acc);
    }
    if (col < cols) part[(int64_t)j * pw + col] = acc;
    else if (col == cols) part[(int64_t)j * pw + D + p.m_max] = M;
    else part[(int64_t)j * pw + D + p.m_max + 1] = acc;
  }
}

// One CTA per (sequence, query head); thread -> output feature.  Merges the
// block partials by their maxima (the global maximum first, by a CTA-wide
// reduction); each chunk's P U_v is multiplied by its V_v,h once, when the
// chunk's last block has been merged.
__global__ void combine_kernel(const __grid_constant__ Params p) {
  __shared__ float pu[kMaxRank];
  __shared__ float red[32];
  const int s = blockIdx.x, jq = blockIdx.y;
  const int d = p.d, pw = d + p.m_max + 2, h = jq / p.g;
  const int c0 = p.seq_chunk[s], c1 = p.seq_chunk[s + 1];
  const int b0 = c0 < p.n_chunks ? p.c[c0].blk0 : p.n_blocks;
  const int b1 = c1 < p.n_chunks ? p.c[c1].blk0 : p.n_blocks;
  const int tid = threadIdx.x, lane = tid & 31, nw = blockDim.x >> 5;
  float M = -INFINITY;
  for (int b = b0 + tid; b < b1; b += blockDim.x) M = fmaxf(M, p.partial[((int64_t)b * p.Hq + jq) * pw + d + p.m_max]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red[tid >> 5] = M;
  __syncthreads();
  M = red[0];
  for (int w = 1; w < nw; ++w) M = fmaxf(M, red[w]);
  const int col = tid;   // blockDim.x == d
  float num = 0.f, den = 0.f;
  for (int ci = c0; ci < c1; ++ci) {
    const ChunkRec& c = p.c[ci];
    const int cb0 = c.blk0, cb1 = c.blk0 + (c.n_tokens + kCta - 1) / kCta;
    float pr = 0.f;   // thread r < rank: this chunk's sum of weighted P U_v, component r
#pragma unroll 4
    for (int b = cb0; b < cb1; ++b) {
      const float* pb = p.partial + ((int64_t)b * p.Hq + jq) * pw;
      const float sc = expf(pb[d + p.m_max] - M);
      num = fmaf(sc, pb[col], num);
      den = fmaf(sc, pb[d + p.m_max + 1], den);
      if (tid < c.rank) pr = fmaf(sc, pb[d + tid], pr);
    }
    if (c.rank > 0) {
      __syncthreads();   // the previous chunk's reads of pu are done
      if (tid < c.rank) pu[tid] = pr;
      __syncthreads();
      const uint16_t* vv = c.vv + ((int64_t)h * d + col) * c.rank;
      float a = 0.f;
      for (int r = 0; r < c.rank; r += 8) {
        const uint4 w = *reinterpret_cast<const uint4*>(vv + r);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          a = fmaf(__uint_as_float(wv[u] << 16), pu[r + 2 * u], a);
          a = fmaf(__uint_as_float(wv[u] & 0xffff0000u), pu[r + 2 * u + 1], a);
        }
      }
      num += a;
    }
  }
  const __nv_bfloat16 o = __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
  p.out[((int64_t)s * p.Hq + jq) * d + col] = *reinterpret_cast<const uint16_t*>(&o);
}

int64_t blocks_of(int32_t n_tokens) { return (n_tokens + kCta - 1) / kCta; }

}  // namespace at
}  // namespace kvrp

using namespace kvrp;

extern "C" {

size_t kv_attend_relocated_workspace_size(int32_t n_chunks, const int32_t* chunk_tokens, int32_t n_q_heads,
                                          int32_t head_dim) {
  if (n_chunks <= 0 || !chunk_tokens || n_q_heads <= 0 || head_dim <= 0) return 0;
  int64_t blocks = 0;
  for (int i = 0; i < n_chunks; ++i) blocks += at::blocks_of(chunk_tokens[i] > 0 ? chunk_tokens[i] : 0);
  const size_t part = sizeof(float) * (size_t)blocks * n_q_heads * (head_dim + at::kMaxRank + 2);
  const size_t qhl = 2 * 2 * (size_t)n_chunks * n_q_heads * head_dim;
  const size_t whl = 2 * 2 * (size_t)n_chunks * n_q_heads * at::kMaxRank;
  return part + qhl + whl + 1024;
}

kvrp_status kv_attend_relocated(const void* q, const kvrp_attn_chunk* chunks, int32_t n_chunks,
                                const int32_t* seq_chunks, int32_t n_seqs, int32_t n_q_heads, int32_t n_kv_heads,
                                int32_t head_dim, double rope_theta, float softmax_scale, void* out,
                                void* workspace, size_t workspace_bytes, kvrp_stream_t stream) {
  if (!q || !chunks || !seq_chunks || !out) return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: NULL argument");
  if (n_chunks <= 0 || n_chunks > at::kMaxChunks)
    return fail(KVRP_ERR_UNSUPPORTED, "kv_attend_relocated: 1 <= n_chunks <= %d", at::kMaxChunks);
  if (n_seqs <= 0 || n_seqs > 65535) return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: 1 <= n_seqs <= 65535");
  if (head_dim != 64 && head_dim != 128)
    return fail(KVRP_ERR_UNSUPPORTED, "kv_attend_relocated: head_dim must be 64 or 128");
  if (n_kv_heads <= 0 || n_q_heads <= 0 || n_q_heads % n_kv_heads || n_q_heads / n_kv_heads > at::kMaxGroup)
    return fail(KVRP_ERR_UNSUPPORTED, "kv_attend_relocated: n_q_heads must be a multiple of n_kv_heads, at most %d x",
                at::kMaxGroup);
  if (!(rope_theta > 0.0) || !std::isfinite(rope_theta) || !(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: rope_theta and softmax_scale must be > 0");
  if (!aligned16(q) || !aligned16(out)) return fail(KVRP_ERR_ALIGNMENT, "kv_attend_relocated: q, out not 16-byte aligned");
  if (seq_chunks[0] != 0 || seq_chunks[n_seqs] != n_chunks)
    return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: seq_chunks must run from 0 to n_chunks");
  std::vector<int32_t> tok(n_chunks);
  int m_max = 0;
  for (int s = 0; s < n_seqs; ++s)
    if (seq_chunks[s + 1] < seq_chunks[s])
      return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: seq_chunks must not decrease");
  for (int i = 0; i < n_chunks; ++i) {
    const kvrp_attn_chunk& c = chunks[i];
    if (c.n_tokens < 0) return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: chunk %d: n_tokens < 0", i);
    if (c.n_tokens > 0 && (!c.k || !c.v)) return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: chunk %d: NULL k/v", i);
    if (c.rank < 0 || c.rank > at::kMaxRank || c.rank % 16)
      return fail(KVRP_ERR_UNSUPPORTED, "kv_attend_relocated: chunk %d: rank must be 0 or a multiple of 16 up to %d", i,
                  at::kMaxRank);
    if (c.rank > 0 && (!c.uk || !c.vk || !c.uv || !c.vv))
      return fail(KVRP_ERR_INVALID_ARG, "kv_attend_relocated: chunk %d: rank > 0 needs all four factors", i);
    if ((c.k && !aligned16(c.k)) || (c.v && !aligned16(c.v)) || (c.uk && !aligned16(c.uk)) || (c.uv && !aligned16(c.uv)) ||
        (c.vk && !aligned16(c.vk)) || (c.vv && !aligned16(c.vv)))
      return fail(KVRP_ERR_ALIGNMENT, "kv_attend_relocated: chunk %d: pointers must be 16-byte aligned", i);
    tok[i] = c.n_tokens;
    m_max = std::max(m_max, (int)c.rank);
  }
  const size_t need = kv_attend_relocated_workspace_size(n_chunks, tok.data(), n_q_heads, head_dim);
  if (!workspace || workspace_bytes < need)
    return fail(KVRP_ERR_WORKSPACE, "kv_attend_relocated: workspace of %zu bytes needed", need);

  static_assert(sizeof(at::Params) <= 32000, "kernel parameter block too large");
  at::Params* pp = new at::Params;   // ~17 KB: off the stack
  std::memset(pp, 0, sizeof(at::Params));
  at::Params& p = *pp;
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255));
  const size_t qhl_bytes = (2 * 2 * (size_t)n_chunks * n_q_heads * head_dim + 255) / 256 * 256;
  const size_t whl_bytes = (2 * 2 * (size_t)n_chunks * n_q_heads * at::kMaxRank + 255) / 256 * 256;
  p.qhl = reinterpret_cast<uint16_t*>(base);
  p.whl = reinterpret_cast<uint16_t*>(base + qhl_bytes);
  p.partial = reinterpret_cast<float*>(base + qhl_bytes + whl_bytes);
  p.n_chunks = n_chunks;
  p.n_seqs = n_seqs;
  p.Hq = n_q_heads;
  p.Hkv = n_kv_heads;
  p.d = head_dim;
  p.g = n_q_heads / n_kv_heads;
  p.scale = softmax_scale;
  p.theta = rope_theta;
  int blk = 0;
  for (int s = 0; s < n_seqs; ++s)
    for (int i = seq_chunks[s]; i < seq_chunks[s + 1]; ++i) {
      const kvrp_attn_chunk& c = chunks[i];
      at::ChunkRec& r = p.c[i];
      r.k = static_cast<const uint16_t*>(c.k);
      r.v = static_cast<const uint16_t*>(c.v);
      r.uk = static_cast<const uint16_t*>(c.uk);
      r.vk = static_cast<const uint16_t*>(c.vk);
      r.uv = static_cast<const uint16_t*>(c.uv);
      r.vv = static_cast<const uint16_t*>(c.vv);
      r.n_tokens = c.n_tokens;
      r.rank = c.rank;
      r.seq = s;
      r.blk0 = blk;
      p.delta[i] = c.delta;
      blk += (int)at::blocks_of(c.n_tokens);
    }
  p.n_blocks = blk;
  for (int s = 0; s <= n_seqs; ++s) p.seq_chunk[s] = seq_chunks[s];
  p.m_max = m_max;

  cudaStream_t st = stream;
  const at::BlockSmem L = at::block_smem(head_dim, m_max);
  void (*blk_fn)(at::Params) = head_dim == 64 ? (m_max <= 32 ? at::block_kernel<64, 4> : at::block_kernel<64, 16>)
                                              : (m_max <= 32 ? at::block_kernel<128, 4> : at::block_kernel<128, 16>);
  cudaError_t e = cudaFuncSetAttribute(blk_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L.bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(at::prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, head_dim * at::kMaxRank * 2);
  if (e == cudaSuccess) {
    at::prep_kernel<<<dim3(n_chunks, n_kv_heads), 256, (size_t)head_dim * m_max * 2, st>>>(p);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess && blk > 0) {
    blk_fn<<<dim3(blk, n_kv_heads), at::kThreads, L.bytes, st>>>(p);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    at::combine_kernel<<<dim3(n_seqs, n_q_heads), head_dim, 0, st>>>(p);   // one thread per feature
    e = cudaGetLastError();
  }
  delete pp;
  if (e != cudaSuccess) return fail(KVRP_ERR_CUDA, "kv_attend_relocated: %s", cudaGetErrorString(e));
  return KVRP_OK;
}

}  // extern "C"
