// Patch formation: the rank-m factors of the conditioning deficit.
//
// Kamera (gist.science/pt/paper/2606.23581, section 2, patch bullet) forms the
// patch once per chunk: a conditioned pass over [A, B] yields KV(B|A), and the
// top-m factors of the deficit come from an SVD.  Here the deficit is taken in
// the destination frame, Delta = KV(B|A) - R(delta) KV(B|empty), so that
// R(delta) KV(B|empty) + U_m V_m^T reproduces KV(B|A) up to the truncation.
// The orbit patch (same page, section 3, reordering bullet) averages the
// deficit over the orderings pi of a cached set before the factorisation:
//   Delta = mean_pi [KV(B|A_pi) - R(delta_pi) KV(B|empty)]
//         = mean_pi KV(B|A_pi) - Rbar KV(B|empty),
// Rbar being the mean of the rotations, itself a per-pair 2x2 matrix of the
// rotate-half form (mean cosine, mean sine), so the canonical cache is read once.
//
// Method (every layer of a call batched in each launch):
//   1. Delta from the bf16 caches, stored in bf16 twice: rows [T][D] and
//      transposed [D][T], so that every product below reads a K-major operand;
//   2. randomized range finder: Y = Delta Omega (Omega: the caller's Gaussian
//      test matrix), q subspace iterations Y <- Delta orth(Delta^T orth(Y));
//   3. Q = orth(Y);  B^T = Delta^T Q;  C = B B^T (k x k);
//   4. C = U_B Lambda U_B^T by parallel cyclic Jacobi; W = U_B[:, :m] Lambda_m^(-1/2);
//   5. V_m = orth(B^T W) (orthonormal right factors), U_m = Delta V_m.
// orth() is shifted Cholesky QR: X <- X R^-1 with R^T R = X^T X + s I, the
// shift s a small multiple of trace(X^T X), one round each time.  After the
// subspace iterations the final Y is conditioned like Delta's top singular values
// (one product past an orthonormal basis), and V_m is orthonormalised again at the
// end, so a second round on Q changes no residual measurably.
//
// The passes over Delta (steps 2, 3 and 5: 2q + 3 of them) are the bulk of the
// work: tall-skinny products with k <= 96 columns, run on the tensor cores by
// pass_kernel (TMA-staged bf16 tiles, tcgen05.mma into a TMEM accumulator,
// fp32 results).  The skinny operands are rounded to bf16 for these products;
// everything else -- the Gram matrices, the k x k solves, the small
// right-multiplies -- stays in fp32 on the CUDA cores (gram_kernel,
// apply_kernel and the one-CTA-per-layer solvers).
#include <cudaTypedefs.h>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "kvrp.h"
#include "kvrp_plan.h"
#include "kvrp_ptx.h"

namespace kvrp {
namespace pf {

constexpr int kMaxK = 96;          // rank + oversampling bound (k x k solves live in shared memory)
constexpr int kMaxOrbit = 64;      // conditioned caches averaged by one call
constexpr int kJacobiSweeps = 2;   // the top-m subspace has settled by then (V_m is re-orthonormalised)
constexpr int kThreads = 256;
constexpr int kJacThreads = 320;   // jacobi_kernel: one 2 x 2 block of A and one row chunk of V^T per thread for k <= 48
constexpr int kTile = 128;         // output rows per pass_kernel CTA
constexpr int kPassStages = 4;     // pass_kernel pipeline depth
constexpr int kPassK = 64;         // pass_kernel: contraction per stage (one 128-byte swizzle row of bf16)
constexpr int kPassThreads = 192;  // producer warp, MMA warp, four epilogue warps
constexpr int kDeltaTokens = 64;   // tokens per delta_kernel tile
constexpr float kShiftFirst = 1e-5f;    // Cholesky QR shift / trace: a basis of unknown conditioning
constexpr float kShiftSecond = 1e-7f;   // a basis already close to orthonormal
using namespace kvrp::ptx;   // mbarrier, TMA, tcgen05 wrappers; kTimeoutCycles bounds every wait

struct TableParam {
  float4 v[kTablePairs];
};

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t f2_to_bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}
__device__ __forceinline__ uint16_t f_to_bf16(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&b);
}

// ---------------------------------------------------------------------------
// 1. Delta = mean_pi cond_pi - Rbar canonical, written as bf16 rows [T][Dp]
//    and bf16 transposed rows [D][Tp].  A CTA takes 64 tokens of one layer and
//    one segment of the row (a rotated head, the rotated MLA tail, or up to 128
//    unrotated features), staged in shared memory for the transposed write.
// ---------------------------------------------------------------------------
struct DeltaArgs {
  const uint16_t* cond[kMaxOrbit];
  const uint16_t* canon;
  uint16_t* out;       // [L][T][Dp]
  uint16_t* out_t;     // [L][D][Tp]
  int64_t cond_stride, canon_stride;   // elements between layers of the inputs
  int n_cond, T, D, Dp, Tp, rope_kind, rot_dim;
  float inv_n;
  float* g_zero;        // the Gram accumulators, zeroed here for the first Gram of the call
  int64_t g_count;      // floats (a multiple of 4)
};

// Segment sg of a row: unrotated features [0, plain_end) in 128-wide pieces,
// then the rotated heads (or the rotated MLA tail).
struct Segment {
  int f0, W;
  bool turns;
};
__host__ __device__ inline int plain_end_of(int rope_kind, int D, int rot) {
  return rope_kind == KVRP_ROPE_MLA_TAIL ? D - rot : (rope_kind == KVRP_ROPE_NONE ? D : 0);
}
__host__ __device__ inline int segment_count(int rope_kind, int D, int rot) {
  const int n_plain = (plain_end_of(rope_kind, D, rot) + 127) / 128;
  const int n_rot = rope_kind == KVRP_ROPE_HEADS ? D / rot : (rope_kind == KVRP_ROPE_MLA_TAIL ? 1 : 0);
  return n_plain + n_rot;
}
__device__ inline Segment segment_of(int sg, int rope_kind, int D, int rot) {
  const int pe = plain_end_of(rope_kind, D, rot);
  const int n_plain = (pe + 127) / 128;
  Segment s;
  s.turns = sg >= n_plain;
  s.f0 = s.turns ? pe + (sg - n_plain) * rot : sg * 128;
  s.W = s.turns ? rot : min(128, pe - s.f0);
  return s;
}

constexpr int kDeltaUnroll = 4;   // narrow path: work units per thread per batch of loads

__device__ __forceinline__ void bf16x8_to_f(const uint4 w, float (&v)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(u[i] << 16);
    v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint4 f_to_bf16x8(const float (&v)[8]) {
  return make_uint4(f2_to_bf16x2(v[0], v[1]), f2_to_bf16x2(v[2], v[3]), f2_to_bf16x2(v[4], v[5]),
                    f2_to_bf16x2(v[6], v[7]));
}

// The transposed tile: 128 feature rows of 64 tokens (128 bytes), the 4-byte
// word index of a row XOR-ed with a multiple of 4 that depends on the row.  A
// warp's 2-byte stores (8 units of 8 or 16 features x 4 tokens) then fall in
// distinct banks, and 8 consecutive tokens of one row stay one aligned 16-byte
// group for the transposed read.
__device__ __forceinline__ int tile_word_swz(int row) { return (((row >> 3) ^ (row >> 6)) & 7) << 2; }
__device__ __forceinline__ int tile_at(int row, int tl) {   // index in halves
  return row * kDeltaTokens + ((((tl >> 1) ^ tile_word_swz(row))) << 1) + (tl & 1);
}

__global__ void __launch_bounds__(kThreads, 3) delta_kernel(const __grid_constant__ DeltaArgs a,
                                                          const __grid_constant__ TableParam tab) {
  pdl_wait();               // the previous kernel's results are visible
  pdl_launch_dependents();  // the next kernel may start launching
  static_assert(kDeltaTokens == 64, "the tile swizzle assumes 32 words per row");
  // phase table, entry i at i + i / 8: the 8 lanes of a 16-byte read phase take
  // entries 8 apart, which would otherwise share one bank group
  __shared__ float4 tb[kTablePairs + kTablePairs / 8];
  __shared__ __align__(16) uint16_t tile[128 * kDeltaTokens];   // bf16 of the deficit, for the transposed rows
  for (int i = threadIdx.x; i < kTablePairs; i += blockDim.x) tb[i + (i >> 3)] = tab.v[i];
  {
    const int64_t cta = blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
    const int64_t n_threads = (int64_t)gridDim.x * gridDim.y * gridDim.z * blockDim.x;
    for (int64_t e = cta * blockDim.x + threadIdx.x; e < a.g_count / 4; e += n_threads)
      reinterpret_cast<float4*>(a.g_zero)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int l = blockIdx.z;
  const int t0 = blockIdx.x * kDeltaTokens;
  const Segment sg = segment_of(blockIdx.y, a.rope_kind, a.D, a.rot_dim);
  uint16_t* out = a.out + (int64_t)l * a.T * a.Dp;
  uint16_t* out_t = a.out_t + (int64_t)l * a.D * a.Tp;
  const uint16_t* canon = a.canon + (int64_t)l * a.canon_stride;
  __syncthreads();
  const int half = sg.W / 2;
  // Wide path: a unit is 8 frequency pairs (elements [e0, e0+8) and their
  // partners [e0+half, ...)), or 16 consecutive unrotated elements, moved as
  // 16-byte vectors.  It needs half (or W) to be a multiple of 8 (16) and the
  // row start 16-byte aligned.
  const bool wide = (sg.turns ? half % 8 == 0 : sg.W % 16 == 0) && a.D % 8 == 0 && sg.f0 % 8 == 0 &&
                    a.canon_stride % 8 == 0 && a.cond_stride % 8 == 0;
  if (wide) {
    // a thread's units (at most kDeltaWide of them) load everything first, then compute
    constexpr int kDeltaWide = 2;
    const int upt = sg.W / 16;
    const int n_units = kDeltaTokens * upt;
    for (int u0 = 0; u0 < n_units; u0 += kDeltaWide * kThreads) {
      uint4 xa[kDeltaWide], xb[kDeltaWide], ca[kDeltaWide], cb[kDeltaWide];
      int tls[kDeltaWide], e0s[kDeltaWide], e1s[kDeltaWide];
#pragma unroll
      for (int b = 0; b < kDeltaWide; ++b) {
        const int u = u0 + b * kThreads + threadIdx.x;
        const int tl = u / upt, w = u - (u / upt) * upt;
        const int t = t0 + tl;
        const bool live = u < n_units && t < a.T;
        tls[b] = live ? tl : -1;
        e0s[b] = sg.turns ? 8 * w : 16 * w;
        e1s[b] = sg.turns ? 8 * w + half : 16 * w + 8;
        xa[b] = xb[b] = ca[b] = cb[b] = make_uint4(0u, 0u, 0u, 0u);
        if (!live) continue;
        const int64_t row = (int64_t)t * a.D + sg.f0;
        xa[b] = *reinterpret_cast<const uint4*>(canon + row + e0s[b]);
        xb[b] = *reinterpret_cast<const uint4*>(canon + row + e1s[b]);
        if (a.n_cond == 1) {
          const uint16_t* c = a.cond[0] + (int64_t)l * a.cond_stride + row;
          ca[b] = *reinterpret_cast<const uint4*>(c + e0s[b]);
          cb[b] = *reinterpret_cast<const uint4*>(c + e1s[b]);
        }
      }
#pragma unroll
      for (int b = 0; b < kDeltaWide; ++b) {
        const int tl = tls[b];
        if (tl < 0) continue;
        const int e0 = e0s[b], e1 = e1s[b];
        const int64_t row = (int64_t)(t0 + tl) * a.D + sg.f0;
        float x0[8], x1[8], c0[8], c1[8];
        bf16x8_to_f(xa[b], x0);
        bf16x8_to_f(xb[b], x1);
        if (a.n_cond == 1) {
          bf16x8_to_f(ca[b], c0);
          bf16x8_to_f(cb[b], c1);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) c0[i] = c1[i] = 0.f;
          for (int p = 0; p < a.n_cond; ++p) {
            const uint16_t* c = a.cond[p] + (int64_t)l * a.cond_stride + row;
            float v0[8], v1[8];
            bf16x8_to_f(*reinterpret_cast<const uint4*>(c + e0), v0);
            bf16x8_to_f(*reinterpret_cast<const uint4*>(c + e1), v1);
#pragma unroll
            for (int i = 0; i < 8; ++i) { c0[i] += v0[i]; c1[i] += v1[i]; }
          }
        }
        float d0[8], d1[8];
        if (sg.turns) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {   // pairs e0 + 2q, e0 + 2q + 1
            const int ti = e0 + 2 * q;
            const float4 hd = tb[ti + (ti >> 3)], tl4 = tb[ti + 1 + ((ti + 1) >> 3)];
            const float a0 = x0[2 * q], a1 = x0[2 * q + 1], b0 = x1[2 * q], b1 = x1[2 * q + 1];
            const float y00 = fmaf(a0, hd.x, -(b0 * hd.z)) + fmaf(a0, tl4.x, -(b0 * tl4.z));
            const float y01 = fmaf(a1, hd.y, -(b1 * hd.w)) + fmaf(a1, tl4.y, -(b1 * tl4.w));
            const float y10 = fmaf(b0, hd.x, a0 * hd.z) + fmaf(b0, tl4.x, a0 * tl4.z);
            const float y11 = fmaf(b1, hd.y, a1 * hd.w) + fmaf(b1, tl4.y, a1 * tl4.w);
            d0[2 * q] = c0[2 * q] * a.inv_n - y00;
            d0[2 * q + 1] = c0[2 * q + 1] * a.inv_n - y01;
            d1[2 * q] = c1[2 * q] * a.inv_n - y10;
            d1[2 * q + 1] = c1[2 * q + 1] * a.inv_n - y11;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) { d0[i] = c0[i] * a.inv_n - x0[i]; d1[i] = c1[i] * a.inv_n - x1[i]; }
        }
        uint16_t* o = out + (int64_t)(t0 + tl) * a.Dp + sg.f0;
        *reinterpret_cast<uint4*>(o + e0) = f_to_bf16x8(d0);
        *reinterpret_cast<uint4*>(o + e1) = f_to_bf16x8(d1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          tile[tile_at(e0 + i, tl)] = f_to_bf16(d0[i]);
          tile[tile_at(e1 + i, tl)] = f_to_bf16(d1[i]);
        }
      }
    }
  } else {
    const int upt = sg.W / 4;                           // two pairs (or four elements) per unit
    const int n_units = kDeltaTokens * upt;
    for (int u0 = 0; u0 < n_units; u0 += kDeltaUnroll * kThreads) {
      // batch of units: issue every load first, then compute
      float2 x0[kDeltaUnroll], x1[kDeltaUnroll], c0[kDeltaUnroll], c1[kDeltaUnroll];
      int e0s[kDeltaUnroll], e1s[kDeltaUnroll], tls[kDeltaUnroll];
#pragma unroll
      for (int b = 0; b < kDeltaUnroll; ++b) {
        const int u = u0 + b * kThreads + threadIdx.x;
        const int tl = u / upt, w = u - (u / upt) * upt;
        const bool live = u < n_units && t0 + tl < a.T;
        const int e0 = sg.turns ? 2 * w : 4 * w;
        const int e1 = sg.turns ? 2 * w + half : 4 * w + 2;
        e0s[b] = e0; e1s[b] = e1; tls[b] = live ? tl : -1;
        x0[b] = x1[b] = c0[b] = c1[b] = make_float2(0.f, 0.f);
        if (!live) continue;
        const int64_t row = (int64_t)(t0 + tl) * a.D + sg.f0;
        x0[b] = bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(canon + row + e0));   // (x_i, x_i+1)
        x1[b] = bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(canon + row + e1));   // their partners
        for (int p = 0; p < a.n_cond; ++p) {
          const uint16_t* c = a.cond[p] + (int64_t)l * a.cond_stride + row;
          const float2 v0 = bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(c + e0));
          const float2 v1 = bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(c + e1));
          c0[b].x += v0.x; c0[b].y += v0.y; c1[b].x += v1.x; c1[b].y += v1.y;
        }
      }
#pragma unroll
      for (int b = 0; b < kDeltaUnroll; ++b) {
        const int tl = tls[b];
        if (tl < 0) continue;
        const int e0 = e0s[b], e1 = e1s[b];
        float2 y0 = x0[b], y1 = x1[b];
        if (sg.turns) {
          // pairs i, i+1 (i = e0): {C_i, C_i+1, S_i, S_i+1}, then tails
          const float4 hd = tb[e0 + (e0 >> 3)], tl4 = tb[e0 + 1 + ((e0 + 1) >> 3)];
          y0.x = fmaf(x0[b].x, hd.x, -(x1[b].x * hd.z)) + fmaf(x0[b].x, tl4.x, -(x1[b].x * tl4.z));
          y0.y = fmaf(x0[b].y, hd.y, -(x1[b].y * hd.w)) + fmaf(x0[b].y, tl4.y, -(x1[b].y * tl4.w));
          y1.x = fmaf(x1[b].x, hd.x, x0[b].x * hd.z) + fmaf(x1[b].x, tl4.x, x0[b].x * tl4.z);
          y1.y = fmaf(x1[b].y, hd.y, x0[b].y * hd.w) + fmaf(x1[b].y, tl4.y, x0[b].y * tl4.w);
        }
        const float d00 = c0[b].x * a.inv_n - y0.x, d01 = c0[b].y * a.inv_n - y0.y;
        const float d10 = c1[b].x * a.inv_n - y1.x, d11 = c1[b].y * a.inv_n - y1.y;
        uint16_t* o = out + (int64_t)(t0 + tl) * a.Dp + sg.f0;
        *reinterpret_cast<uint32_t*>(o + e0) = f2_to_bf16x2(d00, d01);
        *reinterpret_cast<uint32_t*>(o + e1) = f2_to_bf16x2(d10, d11);
        tile[tile_at(e0, tl)] = f_to_bf16(d00); tile[tile_at(e0 + 1, tl)] = f_to_bf16(d01);
        tile[tile_at(e1, tl)] = f_to_bf16(d10); tile[tile_at(e1 + 1, tl)] = f_to_bf16(d11);
      }
    }
  }
  __syncthreads();
  // transposed rows: 8 tokens (16 bytes) per store; tokens past T land in the
  // row padding (Tp rounds T + 1 up to a multiple of 8) and are never read back
  for (int it = threadIdx.x; it < sg.W * (kDeltaTokens / 8); it += blockDim.x) {
    const int f = it / (kDeltaTokens / 8), t8 = 8 * (it - (it / (kDeltaTokens / 8)) * (kDeltaTokens / 8));
    const int t = t0 + t8;
    if (t >= a.T) continue;
    // tokens t8 .. t8 + 7 of row f: one 16-byte group (t8 is a multiple of 8, the
    // swizzle a multiple of 4 words)
    const uint4 w = *reinterpret_cast<const uint4*>(&tile[f * kDeltaTokens + (((t8 >> 1) ^ tile_word_swz(f)) << 1)]);
    *reinterpret_cast<uint4*>(out_t + (int64_t)(sg.f0 + f) * a.Tp + t) = w;
  }
}

// 16 consecutive fp32 TMEM columns of this warp's 32 lanes, completed in the same statement
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Shared-memory matrix descriptor: K-major operand staged by a 128-byte
// swizzled TMA box (rows of 64 bf16 = 128 B, 8-row atoms 1024 B apart).
__device__ __forceinline__ uint64_t desc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused: K stays inside the atom)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: next 8-row atom
  d |= (uint64_t)1 << 46;                      // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;                      // layout: 128-byte swizzle
  return d;
}
// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_bf16_f32(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// ---------------------------------------------------------------------------
// 2. pass_kernel: out[l][r][c] = sum_k A[l][r][k] B[l][c][k] for r < M, c < kp,
//    A and B bf16 K-major (tensor maps with 128-byte swizzled boxes {64, 128}
//    and {64, kp}), fp32 out [L][M][kp].  One CTA per (128-row tile, layer):
//    warp 0 streams the stages with TMA, warp 1 owns the TMEM accumulator and
//    issues tcgen05.mma (M 128, N kp, K 16), warps 2-5 drain TMEM to global.
//    Every wait is bounded; a timeout sets KVRP_DEV_TIMEOUT in *status.
// ---------------------------------------------------------------------------
struct PassArgs {
  float* out;
  int64_t sO;         // out layer stride (elements)
  int M, K, kp;
  int b_layered;      // B has one matrix per layer (else layer 0 for all)
  int kb_per_split;   // contraction blocks of 64 per slice; slices add into a zeroed out
  int splits, layers;
  uint32_t* status;
};

// Bounded wait that ignores the abort flag: lets this CTA's own copies land before it exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint32_t* status) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kTimeoutCycles) {
      if (status) atomicOr(status, KVRP_DEV_TIMEOUT);
      return;
    }
  }
}

// Persistent: CTA i takes items i, i + gridDim.x, ... of (128-row tile, K slice,
// layer).  The producer streams K-blocks through the stage ring without a break
// between items; the MMA warp accumulates item j into TMEM buffer j % 2 while the
// epilogue drains buffer (j - 1) % 2.
__global__ void __launch_bounds__(kPassThreads, 2) pass_kernel(const __grid_constant__ CUtensorMap map_a,
                                                                const __grid_constant__ CUtensorMap map_b,
                                                                PassArgs a) {
  pdl_wait();               // the previous kernel's results are visible
  pdl_launch_dependents();  // the next kernel may start launching
  extern __shared__ __align__(1024) uint8_t smp[];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const uint32_t base = (smem_u32(smp) + 1023u) & ~1023u;
  const uint32_t a_bytes = kTile * kPassK * 2;                 // 16 KiB
  const uint32_t b_bytes = (uint32_t)a.kp * kPassK * 2;        // kp rows of 128 B (a multiple of 1 KiB)
  const uint32_t stage_bytes = a_bytes + b_bytes;
  const uint32_t bars = base + kPassStages * stage_bytes;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (kPassStages + s); };
  auto acc_full = [&](int b) { return bars + 8u * (2 * kPassStages + b); };
  auto acc_empty = [&](int b) { return bars + 8u * (2 * kPassStages + 2 + b); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ncols = a.kp <= 32 ? 32u : a.kp <= 64 ? 64u : 128u;   // one accumulator
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPassStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 4);   // the four epilogue warps
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(2 * ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int tiles = (a.M + kTile - 1) / kTile;
  const int n_items = tiles * a.splits * a.layers;
  const int nkb_all = (a.K + kPassK - 1) / kPassK;
  const bool split = a.splits > 1;
  volatile int* abort_p = &abort_flag;
  struct Item {
    int m0, kb0, nk, l;
  };
  auto item_of = [&](int it) {
    Item r;
    const int t = it % tiles, rest = it / tiles;
    r.m0 = t * kTile;
    r.kb0 = (rest % a.splits) * a.kb_per_split;
    r.l = rest / a.splits;
    r.nk = max(0, min(nkb_all - r.kb0, a.kb_per_split));
    return r;
  };

  if (warp == 0) {
    if (lane == 0) {
      int g = 0;   // K-blocks issued by this CTA
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const Item r = item_of(it);
        const int lb = a.b_layered ? r.l : 0;
        bool ok = true;
        for (int kb = 0; kb < r.nk; ++kb, ++g) {
          const int st = g % kPassStages;
          if (g >= kPassStages && !wait_phase(empty(st), ((g / kPassStages) - 1) & 1, abort_p, a.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + st * stage_bytes;
          mbar_expect_tx(full(st), stage_bytes);
          tma_load_3d(sa, &map_a, full(st), (r.kb0 + kb) * kPassK, r.m0, r.l);
          tma_load_3d(sa + a_bytes, &map_b, full(st), (r.kb0 + kb) * kPassK, 0, lb);
        }
        if (!ok) break;
      }
      // every issued copy must land before the CTA may exit
      for (int q = max(0, g - kPassStages); q < g; ++q) drain_wait(full(q % kPassStages), (q / kPassStages) & 1, a.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(a.kp);
      int g = 0, j = 0;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
        const Item r = item_of(it);
        const int b = j & 1;
        const uint32_t acc = tmem + (uint32_t)b * ncols;
        // the epilogue has drained this buffer (item j - 2)
        if (j >= 2 && !wait_phase(acc_empty(b), ((j >> 1) - 1) & 1, abort_p, a.status)) break;
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < r.nk; ++kb, ++g) {
          const int st = g % kPassStages;
          if (!wait_phase(full(st), (g / kPassStages) & 1, abort_p, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + st * stage_bytes;
#pragma unroll
          for (int q = 0; q < kPassK / 16; ++q)
            mma_bf16(acc, desc_k_sw128(sa + 32u * q), desc_k_sw128(sa + a_bytes + 32u * q), idesc,
                     (kb | q) != 0 ? 1u : 0u);
          mma_commit(empty(st));   // the stage is free once these MMAs have read it
        }
        if (!ok) break;
        mma_commit(acc_full(b));   // arrives when every MMA issued so far has completed
      }
    }
  } else {
    const int quarter = warp & 3;              // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;
    int j = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
      const Item r = item_of(it);
      const int b = j & 1;
      // tcgen05.ld is warp-collective: the whole warp loads or none of it
      const bool ok = __all_sync(0xffffffffu, wait_phase(acc_full(b), (j >> 1) & 1, abort_p, a.status));
      tc_fence_after();
      if (ok && r.nk > 0) {
        float* o = a.out + (int64_t)r.l * a.sO + (int64_t)(r.m0 + row) * a.kp;
        for (int c0 = 0; c0 < a.kp; c0 += 16) {
          float v[16];
          tmem_ld16(tmem + (uint32_t)b * ncols + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
          if (r.m0 + row < a.M) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 f4 = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
              if (split) atomicAdd(reinterpret_cast<float4*>(o + c0 + 4 * q), f4);
              else *reinterpret_cast<float4*>(o + c0 + 4 * q) = f4;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(b));   // this warp is done with buffer b
      if (!ok) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * ncols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// 3. Skinny fp32 products on the CUDA cores (the k x k side of the method).
//    gram_kernel:  G[l] += X[l]^T X[l] over a slice of rows, X [R][KP] fp32;
//                  row slices sized for ~4 CTAs per SM stream through shared
//                  memory in double-buffered stages (cp.async); each value is
//                  split once into a tf32 high part and remainder, and the
//                  product runs on the tensor cores as three tf32 MMAs per tile;
//                  slices add into a zeroed G.
//    apply_kernel: out[l][r] = X[l][r] M[l] (M KP x KP), one thread per row,
//                  M read from shared memory as broadcast float4 rows; with
//                  `solve`, M is chol_kernel's R and out = X R^-1 by
//                  substitution.  Output fp32 rows [R][KP], or bf16 transposed
//                  rows [KP][ldt].
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }


// fp32 -> tf32 (round to nearest, ties away), the value kept in a 32-bit register.
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// D += A B, m16n8k8, tf32 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// G = X^T X on the tensor cores: each fp32 value splits into a tf32 high part and
// a tf32 remainder, and G takes hi.hi + hi.lo + lo.hi (the lo.lo term is below
// fp32 rounding of the sum).  G is symmetric, so only the 16 x 8 output tiles that
// reach the upper triangle are formed (tile (mt, nt) with nt >= 2 mt: 12 of 18 at
// KP = 48); its readers take entry (min(i, j), max(i, j)).  Warp w owns tiles
// w, w + 8, ... of that list and runs every staged row through them.
template <int KP>
__global__ void __launch_bounds__(kThreads) gram_kernel(const float* X, int64_t sX, float* G, int64_t sG, int R,
                                                        int rows_per_cta) {
  pdl_wait();               // the previous kernel's results are visible
  pdl_launch_dependents();  // the next kernel may start launching
  constexpr int MT = KP / 16, NT = KP / 8;
  constexpr int TILES = MT * NT - MT * (MT - 1);   // row mt holds the NT - 2 mt tiles nt >= 2 mt
  constexpr int TPW = (TILES + 7) / 8;             // tiles per warp
  // tile t of the list: its row mt, the first tile of that row S(mt) = mt NT - mt (mt - 1)
  auto tile_of = [](int t, int& m0, int& n0) {
    int mt = 0;
#pragma unroll
    for (int r = 1; r < MT; ++r)
      if (r * NT - r * (r - 1) <= t) mt = r;
    m0 = 16 * mt;
    n0 = 8 * (2 * mt + t - (mt * NT - mt * (mt - 1)));
  };
  constexpr int XP = KP + 8;   // staged row pitch: fragment reads fall in distinct banks
  constexpr int CH = KP <= 48 ? 32 : 16;   // rows per stage (static shared memory < 48 KB)
  __shared__ __align__(16) float xs[2][CH][XP];         // fp32 rows, by cp.async
  __shared__ __align__(16) uint32_t xh[CH][XP], xl[CH][XP];   // their tf32 high parts and remainders
  const int l = blockIdx.y;
  const float* x = X + (int64_t)l * sX;
  const int r0 = blockIdx.x * rows_per_cta;
  const int r1 = min(R, r0 + rows_per_cta);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  auto load = [&](int buf, int c0) {
    for (int ch = tid; ch < CH * KP / 4; ch += kThreads) {
      const int r = ch / (KP / 4), c4 = (ch - r * (KP / 4)) * 4;
      const bool ok = c0 + r < r1;
      cp_async16(&xs[buf][r][c4], ok ? x + (int64_t)(c0 + r) * KP + c4 : x, ok);
    }
    cp_async_commit();
  };
  float acc[TPW][4] = {};
  const int n_chunks = (r1 - r0 + CH - 1) / CH;
  if (n_chunks > 0) load(0, r0);
  for (int c = 0; c < n_chunks; ++c) {
    if (c + 1 < n_chunks) {
      load((c + 1) & 1, r0 + (c + 1) * CH);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    // split every staged value once (rows past r1 are zero)
    for (int e = tid; e < CH * KP; e += kThreads) {
      const int r = e / KP, k = e - r * KP;
      const float v = xs[c & 1][r][k];
      const uint32_t h = to_tf32(v);
      xh[r][k] = h;
      xl[r][k] = to_tf32(v - __uint_as_float(h));
    }
    __syncthreads();
#pragma unroll
    for (int k0 = 0; k0 < CH; k0 += 8) {
#pragma unroll
      for (int i = 0; i < TPW; ++i) {
        const int t = warp + 8 * i;
        if (t >= TILES) break;
        int m0, n0;
        tile_of(t, m0, n0);
        // A = X^T (rows m, columns k), B = X (rows k, columns n)
        const uint32_t ah[4] = {xh[k0 + tig][m0 + gid], xh[k0 + tig][m0 + gid + 8], xh[k0 + tig + 4][m0 + gid],
                                xh[k0 + tig + 4][m0 + gid + 8]};
        const uint32_t al[4] = {xl[k0 + tig][m0 + gid], xl[k0 + tig][m0 + gid + 8], xl[k0 + tig + 4][m0 + gid],
                                xl[k0 + tig + 4][m0 + gid + 8]};
        mma_tf32(acc[i], al, xh[k0 + tig][n0 + gid], xh[k0 + tig + 4][n0 + gid]);
        mma_tf32(acc[i], ah, xl[k0 + tig][n0 + gid], xl[k0 + tig + 4][n0 + gid]);
        mma_tf32(acc[i], ah, xh[k0 + tig][n0 + gid], xh[k0 + tig + 4][n0 + gid]);
      }
    }
    __syncthreads();   // the split arrays and this stage buffer are reused
  }
  float* g = G + (int64_t)l * sG;
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    const int t = warp + 8 * i;
    if (t >= TILES) break;
    int m0, n0;
    tile_of(t, m0, n0);
#pragma unroll
    for (int e = 0; e < 4; ++e) atomicAdd(&g[(m0 + gid + (e >> 1) * 8) * KP + n0 + 2 * tig + (e & 1)], acc[i][e]);
  }
}

template <int KP>
__global__ void __launch_bounds__(128) apply_kernel(const float* X, int64_t sX, const float* M, int64_t sM, float* out,
                                                    int64_t sO, uint16_t* out_t, int64_t sT, int ldt, int R, int solve) {
  pdl_wait();               // the previous kernel's results are visible
  pdl_launch_dependents();  // the next kernel may start launching
  __shared__ __align__(16) float ms[KP][KP];
  const int l = blockIdx.y;
  const float* m = M + (int64_t)l * sM;
  for (int e = threadIdx.x; e < KP * KP / 4; e += blockDim.x)
    reinterpret_cast<float4*>(&ms[0][0])[e] = reinterpret_cast<const float4*>(m)[e];
  __syncthreads();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  const float* x = X + (int64_t)l * sX + (int64_t)r * KP;
  float xv[KP], o[KP];
#pragma unroll
  for (int i = 0; i < KP; i += 4) {
    const float4 v = *reinterpret_cast<const float4*>(x + i);
    xv[i] = v.x; xv[i + 1] = v.y; xv[i + 2] = v.z; xv[i + 3] = v.w;
  }
  if (solve) {
    // o R = x with R from chol_kernel (diagonal held as 1 / R_jj): o_j = x_j / R_jj, then
    // x_l -= o_j R_jl for l > j (right-looking substitution: short dependency chains)
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      o[j] = xv[j] * ms[j][j];
      const int l4 = (j + 4) & ~3;   // first 16-byte aligned column after j
#pragma unroll
      for (int l = j + 1; l < l4 && l < KP; ++l) xv[l] = fmaf(-o[j], ms[j][l], xv[l]);
#pragma unroll
      for (int l = l4; l < KP; l += 4) {   // the rest of row j as broadcast float4 reads
        const float4 mv = *reinterpret_cast<const float4*>(&ms[j][l]);
        xv[l] = fmaf(-o[j], mv.x, xv[l]);
        xv[l + 1] = fmaf(-o[j], mv.y, xv[l + 1]);
        xv[l + 2] = fmaf(-o[j], mv.z, xv[l + 2]);
        xv[l + 3] = fmaf(-o[j], mv.w, xv[l + 3]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < KP; ++j) o[j] = 0.f;
#pragma unroll
    for (int i = 0; i < KP; ++i) {
#pragma unroll
      for (int j4 = 0; j4 < KP; j4 += 4) {
        const float4 mv = *reinterpret_cast<const float4*>(&ms[i][j4]);
        o[j4] = fmaf(xv[i], mv.x, o[j4]);
        o[j4 + 1] = fmaf(xv[i], mv.y, o[j4 + 1]);
        o[j4 + 2] = fmaf(xv[i], mv.z, o[j4 + 2]);
        o[j4 + 3] = fmaf(xv[i], mv.w, o[j4 + 3]);
      }
    }
  }
  if (out_t) {
    uint16_t* ot = out_t + (int64_t)l * sT + r;
#pragma unroll
    for (int j = 0; j < KP; ++j) ot[(int64_t)j * ldt] = f_to_bf16(o[j]);
  } else {
    float* op = out + (int64_t)l * sO + (int64_t)r * KP;
#pragma unroll
    for (int j = 0; j < KP; j += 4) *reinterpret_cast<float4*>(op + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
  }
}

// Sum of one value per thread over the CTA (blockDim.x == kThreads); `scratch`
// holds kThreads / 32 floats.  Every thread gets the total.
template <int NT = kThreads>   // threads of the CTA; scratch holds NT / 32 floats
__device__ __forceinline__ float block_sum(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) t += scratch[w];
  __syncthreads();
  return t;
}

// ---------------------------------------------------------------------------
// 4. Shifted Cholesky of a Gram matrix, fp32, one CTA per layer:
//    R^T R = G + s I (s = rel * trace G); out = R with its diagonal stored as
//    1 / R_jj, zero outside the leading k x k block (apply_kernel's solve mode
//    then forms X R^-1 by substitution, so R is never inverted).
//    Blocked right-looking factorisation over 16 x 16 blocks, in place in
//    shared memory (entries past k hold the identity, which never couples to
//    the leading block): warp 0 factors the diagonal block warp-synchronously,
//    one thread per column solves the block row of R from it, and all threads
//    apply the rank-16 update to the trailing matrix in 2 x 2 register tiles.
//    Three CTA barriers per block instead of one per column.
// ---------------------------------------------------------------------------
template <int KP>
__global__ void __launch_bounds__(kThreads) chol_kernel(float* G, int64_t sG, float* Rf, int64_t sR,
                                                                 int k, float rel) {
  pdl_wait();               // the previous kernel's results are visible
  pdl_launch_dependents();  // the next kernel may start launching
  constexpr int P = KP + 1;    // row pitch: neighbouring rows start in different banks
  constexpr int NB = KP / 16;
  __shared__ float A[KP * P];
  __shared__ float scratch[kThreads / 32];
  __shared__ float rdiag[KP];
  float* g = G + (int64_t)blockIdx.x * sG;
  float* out = Rf + (int64_t)blockIdx.x * sR;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float tr = 0.f;
  for (int e = tid; e < KP * KP; e += kThreads) {
    const int i = e / KP, j = e - i * KP;
    const float v = (i < k && j < k) ? g[min(i, j) * KP + max(i, j)] : (i == j ? 1.f : 0.f);   // the upper triangle
    A[i * P + j] = v;
    if (i == j && i < k) tr += v;
  }
  tr = block_sum(tr, scratch);   // (its barriers: every thread has read G)
  for (int e = tid; e < KP * KP; e += kThreads) g[e] = 0.f;   // zeroed for the next Gram
  const float shift = tr > 0.f ? rel * tr : 1e-30f;
  if (tid < k) A[tid * P + tid] += shift;
  __syncthreads();
  for (int b = 0; b < NB; ++b) {
    const int o = 16 * b;
    if (warp == 0) {
      // diagonal block in registers: lane l holds column l of the block (lanes
      // 16 .. 31 repeat lanes 0 .. 15 and store nothing); its upper triangle
      // becomes R_bb, row j of R coming from lane j's column by shuffles
      const int l = lane & 15;
      float col[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) col[r] = A[(o + r) * P + o + l];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float d = fmaxf(__shfl_sync(0xffffffffu, col[j], j), shift);
        const float rs = rsqrtf(d);
        col[j] = l > j ? col[j] * rs : (l == j ? d * rs : col[j]);   // R[j][l]
#pragma unroll
        for (int r = 1; r < 16; ++r) {   // r > j; a fixed trip count keeps col[] in registers
          if (r <= j) continue;
          const float rjr = __shfl_sync(0xffffffffu, col[j], r);     // R[j][r], from lane r
          if (l >= r) col[r] = fmaf(-rjr, col[j], col[r]);
        }
        if (lane == j) rdiag[o + j] = rs;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (lane < 16 && l >= r) A[(o + r) * P + o + l] = col[r];
    }
    __syncthreads();
    const int nt = KP - o - 16;                              // columns right of the block
    if (tid < nt) {
      // block row of R: R_bb^T x = A[o .. o + 16)[c], forward substitution
      const int c = o + 16 + tid;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = A[(o + i) * P + c];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float v = x[i];
#pragma unroll
        for (int j = 0; j < 15; ++j)
          if (j < i) v = fmaf(-A[(o + j) * P + o + i], x[j], v);
        x[i] = v * rdiag[o + i];
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) A[(o + i) * P + c] = x[i];
    }
    __syncthreads();
    // trailing update A[r][c] -= sum_i R[o+i][r] R[o+i][c], r, c >= o + 16 (both triangles)
    const int h = nt / 2;
    for (int t = tid; t < h * h; t += kThreads) {
      const int r = o + 16 + 2 * (t / h), c = o + 16 + 2 * (t % h);
      float a00 = A[r * P + c], a01 = A[r * P + c + 1], a10 = A[(r + 1) * P + c], a11 = A[(r + 1) * P + c + 1];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float* row = A + (o + i) * P;
        const float u0 = row[r], u1 = row[r + 1], v0 = row[c], v1 = row[c + 1];
        a00 = fmaf(-u0, v0, a00);
        a01 = fmaf(-u0, v1, a01);
        a10 = fmaf(-u1, v0, a10);
        a11 = fmaf(-u1, v1, a11);
      }
      A[r * P + c] = a00;
      A[r * P + c + 1] = a01;
      A[(r + 1) * P + c] = a10;
      A[(r + 1) * P + c + 1] = a11;
    }
    __syncthreads();
  }
  // R row by row, its diagonal stored as 1 / R_jj (zero outside the leading k x k block)
  for (int e = tid; e < KP * KP; e += kThreads) {
    const int i = e / KP, j = e - i * KP;
    out[e] = (i < k && j < k && j >= i) ? (i == j ? rdiag[i] : A[i * P + j]) : 0.f;
  }
}

// ---------------------------------------------------------------------------
// 5. Symmetric eigenproblem C = U L U^T by parallel cyclic Jacobi (round-robin
//    pairing: n/2 disjoint rotations per step), fp32, one CTA per layer.  A
//    step applies A <- J^T A J as independent 2 x 2 blocks (rows of one pair
//    against columns of another; blocks on or above the diagonal, mirrored),
//    so each thread updates whole blocks with no barrier between the row and
//    column halves of the rotations.  Writes W [kp][kp]: column r < m is the
//    eigenvector of the r-th largest eigenvalue scaled by lambda^(-1/2) (zero
//    where lambda vanishes); other columns zero.
// ---------------------------------------------------------------------------
template <int NT>   // threads per CTA
__global__ void __launch_bounds__(NT) jacobi_kernel(float* Cm, int64_t sC, float* W, int64_t sW, int k, int kp,
                                                    int m) {
  pdl_wait();               // the previous kernel's results are visible
  pdl_launch_dependents();  // the next kernel may start launching
  extern __shared__ __align__(16) float smj[];
  const int P = kp + 1;     // A's row pitch: neighbouring rows start in different banks
  const int PV = kp + 4;    // V^T's row pitch: rows 16-byte aligned for float4 access
  float* A = smj;
  float* VT = smj + (kp * P + 3) / 4 * 4;   // V^T: row r is column r of the accumulated rotations
  __shared__ int4 rot[kMaxK / 2];      // {p, q, cos, sin} of each pair of the step
  __shared__ int order[kMaxK];
  __shared__ float scratch[NT / 32];
  __shared__ int rotated;
  float* c = Cm + (int64_t)blockIdx.x * sC;
  float* w = W + (int64_t)blockIdx.x * sW;
  const int tid = threadIdx.x;
  float ss = 0.f;
  for (int e = tid; e < kp * kp; e += NT) {
    const int i = e / kp, j = e - (e / kp) * kp;
    const float v = (i < k && j < k) ? c[min(i, j) * kp + max(i, j)] : 0.f;   // the upper triangle
    A[i * P + j] = v;
    VT[i * PV + j] = i == j ? 1.f : 0.f;
    ss += v * v;
  }
  // entries below floor_abs are rounding noise of the fp32 input
  const float floor_abs = 1e-6f * sqrtf(block_sum<NT>(ss, scratch));   // (its barriers: every thread has read C)
  for (int e = tid; e < kp * kp; e += NT) c[e] = 0.f;           // zeroed for the next Gram
  const int n2 = k + (k & 1);      // index k (< kp when k is odd) is a dummy that never turns
  const int np = n2 / 2;
  // this thread's 2 x 2 blocks (t1 <= t2), the same at every step
  constexpr int kMaxBlk = ((kMaxK / 2) * (kMaxK / 2 + 1) / 2 + NT - 1) / NT;
  int blk[kMaxBlk];
  int nb = 0;
  {
    int idx = 0;
    for (int t1 = 0; t1 < np; ++t1)
      for (int t2 = t1; t2 < np; ++t2, ++idx)
        if (idx % NT == tid && nb < kMaxBlk) blk[nb++] = (t1 << 8) | t2;
  }
  // V <- V J is V^T <- J^T V^T: rows p and q of V^T, in float4 chunks; this thread's
  // (pair, chunk) items, the same at every step
  const int nch = (k + 3) / 4;
  constexpr int kMaxVit = ((kMaxK / 2) * (kMaxK / 4) + NT - 1) / NT;
  int vit[kMaxVit];
  int nv = 0;
  for (int it = tid; it < np * nch && nv < kMaxVit; it += NT) vit[nv++] = ((it / nch) << 8) | (4 * (it % nch));
  for (int sweep = 0; sweep < kJacobiSweeps; ++sweep) {
    if (tid == 0) rotated = 0;
    __syncthreads();
    for (int step = 0; step < n2 - 1; ++step) {
      if (tid < np) {
        // circle method: player n2-1 stays, the others move one seat per step
        // (step + tid and step - tid + n2 - 1 lie in [0, 2 (n2 - 1)): one wrap each)
        int p = n2 - 1, q = step;
        if (tid > 0) {
          p = step + tid;
          if (p >= n2 - 1) p -= n2 - 1;
          q = step - tid + n2 - 1;
          if (q >= n2 - 1) q -= n2 - 1;
        }
        if (p > q) { const int x = p; p = q; q = x; }
        float cc = 1.f, s = 0.f;
        if (q < k) {
          const float apq = A[p * P + q];
          const float app = A[p * P + p], aqq = A[q * P + q];
          // Any angle gives an exact orthogonal update, so approximate reciprocals
          // and square roots only affect how fast the sweep converges.
          // |a_pq| below 1e-4 sqrt(a_pp a_qq) moves an eigenvector by ~1e-4: the
          // orthonormalisation of B^T W that follows absorbs that
          if (fabsf(apq) > floor_abs && apq * apq > 1e-8f * fabsf(app * aqq)) {
            const float th = __fdividef(aqq - app, 2.f * apq);
            const float r2 = fmaf(th, th, 1.f);
            const float tt = copysignf(__fdividef(1.f, fabsf(th) + r2 * rsqrtf(r2)), th);
            cc = rsqrtf(fmaf(tt, tt, 1.f));
            s = tt * cc;
            if (s != 0.f) rotated = 1;
          }
        }
        rot[tid] = make_int4(p, q, __float_as_int(cc), __float_as_int(s));
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kMaxBlk; ++u) {
        if (u >= nb) break;
        const int t1 = blk[u] >> 8, t2 = blk[u] & 0xFF;
        const int4 r1 = rot[t1], r2 = rot[t2];
        const float s1 = __int_as_float(r1.w), s2 = __int_as_float(r2.w);
        if (s1 == 0.f && s2 == 0.f) continue;
        const float c1 = __int_as_float(r1.z), c2 = __int_as_float(r2.z);
        const int p1 = r1.x, q1 = r1.y, p2 = r2.x, q2 = r2.y;
        const float a = A[p1 * P + p2], b = A[p1 * P + q2], cq = A[q1 * P + p2], d = A[q1 * P + q2];
        // rows: [p1; q1] <- [c1 -s1; s1 c1] [p1; q1]
        const float ra = c1 * a - s1 * cq, rb = c1 * b - s1 * d;
        const float rc = s1 * a + c1 * cq, rd = s1 * b + c1 * d;
        // columns: [p2 q2] <- [p2 q2] [c2 s2; -s2 c2]
        float na = c2 * ra - s2 * rb, nb2 = s2 * ra + c2 * rb;
        float nc = c2 * rc - s2 * rd, nd = s2 * rc + c2 * rd;
        if (t1 == t2) {
          if (s1 != 0.f) { nb2 = 0.f; nc = 0.f; }   // the rotation annihilates a_pq
          A[p1 * P + p2] = na; A[p1 * P + q2] = nb2; A[q1 * P + p2] = nc; A[q1 * P + q2] = nd;
        } else {
          A[p1 * P + p2] = na; A[p1 * P + q2] = nb2; A[q1 * P + p2] = nc; A[q1 * P + q2] = nd;
          A[p2 * P + p1] = na; A[q2 * P + p1] = nb2; A[p2 * P + q1] = nc; A[q2 * P + q1] = nd;
        }
      }
#pragma unroll
      for (int u = 0; u < kMaxVit; ++u) {
        if (u >= nv) break;
        const int4 r = rot[vit[u] >> 8];
        const float s = __int_as_float(r.w);
        if (s == 0.f) continue;
        const float cc = __int_as_float(r.z);
        const int c4 = vit[u] & 0xFF;
        float4* vp = reinterpret_cast<float4*>(VT + r.x * PV + c4);
        float4* vq = reinterpret_cast<float4*>(VT + r.y * PV + c4);
        const float4 a = *vp, b = *vq;
        *vp = make_float4(cc * a.x - s * b.x, cc * a.y - s * b.y, cc * a.z - s * b.z, cc * a.w - s * b.w);
        *vq = make_float4(s * a.x + cc * b.x, s * a.y + cc * b.y, s * a.z + cc * b.z, s * a.w + cc * b.w);
      }
      __syncthreads();
    }
    if (!rotated) break;
    __syncthreads();
  }
  // descending order by rank counting (ties by index).  A NaN diagonal (NaN in the caller's
  // caches) ranks below every number: the comparison stays a strict total order, so the
  // ranks are a permutation of 0 .. k - 1 and every order[] entry read below is set.
  if (tid < k) {
    const float di = A[tid * P + tid];
    const float li = isnan(di) ? -INFINITY : di;
    int rank = 0;
    for (int j = 0; j < k; ++j) {
      const float dj = A[j * P + j];
      const float lj = isnan(dj) ? -INFINITY : dj;
      rank += (lj > li) || (lj == li && j < tid);
    }
    order[rank] = tid;
  }
  __syncthreads();
  const float lmax = fmaxf(A[order[0] * P + order[0]], 0.f);
  for (int e = tid; e < kp * kp; e += NT) {
    const int i = e / kp, r = e - (e / kp) * kp;
    float v = 0.f;
    if (i < k && r < m && r < k) {
      const int o = order[r];
      const float lam = A[o * P + o];
      if (lam > 1e-10f * lmax && lam > 0.f) v = VT[o * PV + i] * rsqrtf(lam);
    }
    w[e] = v;
  }
}

// ---------------------------------------------------------------------------
// 6. Small helpers: Omega^T in bf16, the caller's factors in bf16
// ---------------------------------------------------------------------------
// dst [kp][Dp] bf16 = Omega^T, zero beyond the k columns of Omega [D][k]
__global__ void omega_t_kernel(const float* src, int D, int k, uint16_t* dst, int kp, int Dp) {
  pdl_wait();               // the previous kernel's results are visible
  pdl_launch_dependents();  // the next kernel may start launching
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < kp * D; e += gridDim.x * blockDim.x) {
    const int c = e / D, f = e - (e / D) * D;
    dst[(int64_t)c * Dp + f] = f_to_bf16(c < k ? src[(int64_t)f * k + c] : 0.f);
  }
}
// u_out[l][t][c] = bf16(U[l][t][c]) for c < m, from fp32 [L][T][kp]
__global__ void u_out_kernel(const float* src, int64_t src_stride, int kp, uint16_t* dst, int64_t dst_stride, int rows,
                             int m) {
  pdl_wait();               // the previous kernel's results are visible
  pdl_launch_dependents();  // the next kernel may start launching
  const int l = blockIdx.y;
  const int64_t n = (int64_t)rows * m;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / m;
    const int c = (int)(e - r * m);
    dst[l * dst_stride + e] = f_to_bf16(src[l * src_stride + r * kp + c]);
  }
}
// v_out[l][f][c] = V^T[l][c][f] for c < m, from bf16 [L][kp][ld]
__global__ void v_out_kernel(const uint16_t* src, int64_t src_stride, int ld, uint16_t* dst, int64_t dst_stride, int D,
                             int m) {
  pdl_wait();               // the previous kernel's results are visible
  pdl_launch_dependents();  // the next kernel may start launching
  const int l = blockIdx.y;
  const int64_t n = (int64_t)D * m;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t f = e / m;
    const int c = (int)(e - f * m);
    dst[l * dst_stride + e] = src[l * src_stride + (int64_t)c * ld + f];
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
int64_t round8(int64_t v) { return (v + 7) / 8 * 8; }
int pad16(int k) { return (k + 15) / 16 * 16; }

struct Buffers {
  uint16_t *delta, *delta_t, *st_t, *st_d, *omega_t;   // bf16
  float *y, *y2, *z, *z2, *g, *rfac, *w;               // fp32
  int64_t Dp, Tp, s_delta, s_delta_t, s_st_t, s_st_d, s_tk, s_dk, s_kk;
  size_t bytes;
};

Buffers layout(uint8_t* base, int L, int T, int D, int kp) {
  Buffers b;
  b.Dp = round8(D);
  b.Tp = round8(T + 1);   // room for the odd-token pad of the transposed writes
  b.s_delta = (int64_t)T * b.Dp;
  b.s_delta_t = (int64_t)D * b.Tp;
  b.s_st_t = (int64_t)kp * b.Tp;
  b.s_st_d = (int64_t)kp * b.Dp;
  b.s_tk = (int64_t)T * kp;
  b.s_dk = (int64_t)D * kp;
  b.s_kk = (int64_t)kp * kp;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = (off + bytes + 1023) / 1024 * 1024;
    return base + o;
  };
  b.delta = reinterpret_cast<uint16_t*>(take(2 * (size_t)b.s_delta * L));
  b.delta_t = reinterpret_cast<uint16_t*>(take(2 * (size_t)b.s_delta_t * L));
  b.st_t = reinterpret_cast<uint16_t*>(take(2 * (size_t)b.s_st_t * L));
  b.st_d = reinterpret_cast<uint16_t*>(take(2 * (size_t)b.s_st_d * L));
  b.omega_t = reinterpret_cast<uint16_t*>(take(2 * (size_t)b.s_st_d));
  b.y = reinterpret_cast<float*>(take(4 * (size_t)b.s_tk * L));
  b.y2 = reinterpret_cast<float*>(take(4 * (size_t)b.s_tk * L));
  b.z = reinterpret_cast<float*>(take(4 * (size_t)b.s_dk * L));
  b.z2 = reinterpret_cast<float*>(take(4 * (size_t)b.s_dk * L));
  b.g = reinterpret_cast<float*>(take(4 * (size_t)b.s_kk * L));
  b.rfac = reinterpret_cast<float*>(take(4 * (size_t)b.s_kk * L));
  b.w = reinterpret_cast<float*>(take(4 * (size_t)b.s_kk * L));
  b.bytes = off;
  return b;
}

// 16-significant-bit head of a value (its fp32 tail is value - head)
float head16(double v) {
  if (v == 0.0) return 0.0f;
  int e = 0;
  const double m = std::frexp(v, &e);
  return static_cast<float>(std::ldexp(std::nearbyint(std::ldexp(m, 16)), e - 16));
}

// Mean rotation over the orbit: pair i holds (mean cos(delta_pi theta_i), mean sin(...)),
// computed in fp64 and laid out like the relocation tables (two pairs per
// float4: heads {C_i, C_i+1, S_i, S_i+1}, then the fp32 tails).
void mean_table(const int64_t* deltas, int n, double theta, int rot_dim, float4* tab) {
  float hc[kTablePairs] = {}, hs[kTablePairs] = {}, tc[kTablePairs] = {}, ts[kTablePairs] = {};
  for (int i = 0; i < rot_dim / 2; ++i) {
    const double inv = std::pow(theta, -2.0 * i / rot_dim);
    double c = 0.0, s = 0.0;
    for (int p = 0; p < n; ++p) {
      const double phi = static_cast<double>(deltas[p]) * inv;
      c += std::cos(phi);
      s += std::sin(phi);
    }
    c /= n;
    s /= n;
    hc[i] = head16(c);
    hs[i] = head16(s);
    tc[i] = static_cast<float>(c - hc[i]);
    ts[i] = static_cast<float>(s - hs[i]);
  }
  for (int j = 0; j < kTablePairs / 2; ++j) {
    tab[2 * j] = make_float4(hc[2 * j], hc[2 * j + 1], hs[2 * j], hs[2 * j + 1]);
    tab[2 * j + 1] = make_float4(tc[2 * j], tc[2 * j + 1], ts[2 * j], ts[2 * j + 1]);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 [layers][rows][K] with row pitch `ld` elements, boxes {64, box_rows}, 128-byte swizzle
bool encode_kmajor(CUtensorMap* map, const uint16_t* base, int K, int rows, int layers, int64_t ld,
                   int64_t layer_stride, int box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)layers};
  const cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)layer_stride * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kPassK, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t pass_smem_bytes(int kp) { return 1024 + (size_t)kPassStages * (kTile * kPassK * 2 + kp * kPassK * 2) + 128; }

// Launch with programmatic stream serialization: the kernel may start while the
// previous one on the stream drains, and waits for it in pdl_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

class Runner {
 public:
  Runner(cudaStream_t st, int L, int kp, int sms, uint32_t* status)
      : st_(st), L_(L), kp_(kp), sms_(sms), status_(status) {}
  cudaError_t err = cudaSuccess;
  bool map_fail = false;

  // out[L][M][kp] fp32 = A[L][M][K] B[Lb][kp][K]^T on the tensor cores
  void pass(const uint16_t* A, int64_t a_ld, int64_t a_stride, const uint16_t* B, int64_t b_ld, int64_t b_stride,
            bool b_layered, float* out, int64_t sO, int M, int K) {
    if (err != cudaSuccess || map_fail) return;
    CUtensorMap ma, mb;
    if (!encode_kmajor(&ma, A, K, M, L_, a_ld, a_stride, kTile) ||
        !encode_kmajor(&mb, B, K, kp_, b_layered ? L_ : 1, b_ld, b_stride, kp_)) {
      map_fail = true;
      return;
    }
    // Contraction slices: when tiles x layers cannot fill the resident CTA
    // slots (2 per SM), split K, each slice keeping >= 8 blocks of 64.
    const int tiles = (M + kTile - 1) / kTile;
    const int nkb = (K + kPassK - 1) / kPassK;
    const int cap = 2 * sms_;
    int splits = 1, per = nkb;
    double best = -1.0;
    for (int sp = 1; sp <= std::max(1, nkb / 8); ++sp) {
      const int pr = (nkb + sp - 1) / sp;
      const int n = (nkb + pr - 1) / pr;
      if (n != sp) continue;
      const int64_t total = (int64_t)tiles * L_ * n;
      const int64_t waves = (total + cap - 1) / cap;
      const double score = (double)total / (double)(waves * cap) - 0.01 * n;
      if (score > best + 1e-9) { best = score; splits = n; per = pr; }
    }
    if (splits > 1) {
      err = cudaMemsetAsync(out, 0, sizeof(float) * (size_t)(sO * (L_ - 1) + (int64_t)M * kp_), st_);
      if (err != cudaSuccess) return;
    }
    PassArgs pa{out, sO, M, K, kp_, b_layered ? 1 : 0, per, splits, L_, status_};
    // as many CTAs as keep the item rounds the same, each taking an equal number of items:
    // 448 items on 304 slots still take two rounds, so 224 CTAs do them and the other SMs
    // stay free for concurrent work (another call's solves)
    const int items = tiles * splits * L_;
    const int rounds = (items + cap - 1) / cap;
    err = launch_pdl(pass_kernel, dim3((items + rounds - 1) / rounds), dim3(kPassThreads), pass_smem_bytes(kp_), st_, ma,
                     mb, pa);
  }

  // G[L][kp][kp] = X^T X for X [L][R][kp]
  void gram(const float* X, int64_t sX, float* G, int R) {
    if (err != cudaSuccess) return;
    const int64_t skk = (int64_t)kp_ * kp_;
    // G is zero here: the deficit kernel clears it, and every reader of a Gram (the Cholesky
    // and Jacobi kernels) clears it after reading
    // row slices sized for about four CTAs per SM over all layers (64-row multiples, 64..512)
    const int64_t want = ((int64_t)R * L_ + 4 * sms_ - 1) / (4 * sms_);
    const int rows = (int)std::min<int64_t>(512, std::max<int64_t>(64, (want + 63) / 64 * 64));
    const dim3 grid((R + rows - 1) / rows, L_);
    switch (kp_) {
      case 16: err = launch_pdl(gram_kernel<16>, dim3(grid), dim3(kThreads), 0, st_, X, sX, G, skk, R, rows); break;
      case 32: err = launch_pdl(gram_kernel<32>, dim3(grid), dim3(kThreads), 0, st_, X, sX, G, skk, R, rows); break;
      case 48: err = launch_pdl(gram_kernel<48>, dim3(grid), dim3(kThreads), 0, st_, X, sX, G, skk, R, rows); break;
      case 64: err = launch_pdl(gram_kernel<64>, dim3(grid), dim3(kThreads), 0, st_, X, sX, G, skk, R, rows); break;
      case 80: err = launch_pdl(gram_kernel<80>, dim3(grid), dim3(kThreads), 0, st_, X, sX, G, skk, R, rows); break;
      case 96: err = launch_pdl(gram_kernel<96>, dim3(grid), dim3(kThreads), 0, st_, X, sX, G, skk, R, rows); break;
      default: err = cudaErrorInvalidValue; return;
    }
    err = cudaGetLastError();
  }

  // out[L][R][kp] = X[L][R][kp] M[L][kp][kp] (fp32 rows), or bf16 transposed rows into out_t
  void apply(const float* X, int64_t sX, const float* M, float* out, int64_t sO, int R, bool solve,
             uint16_t* out_t = nullptr, int64_t sT = 0, int ldt = 0) {
    if (err != cudaSuccess) return;
    const int64_t skk = (int64_t)kp_ * kp_;
    const dim3 grid((R + 127) / 128, L_);
    const int up = solve ? 1 : 0;
    switch (kp_) {
      case 16: err = launch_pdl(apply_kernel<16>, dim3(grid), dim3(128), 0, st_, X, sX, M, skk, out, sO, out_t, sT, ldt, R, up); break;
      case 32: err = launch_pdl(apply_kernel<32>, dim3(grid), dim3(128), 0, st_, X, sX, M, skk, out, sO, out_t, sT, ldt, R, up); break;
      case 48: err = launch_pdl(apply_kernel<48>, dim3(grid), dim3(128), 0, st_, X, sX, M, skk, out, sO, out_t, sT, ldt, R, up); break;
      case 64: err = launch_pdl(apply_kernel<64>, dim3(grid), dim3(128), 0, st_, X, sX, M, skk, out, sO, out_t, sT, ldt, R, up); break;
      case 80: err = launch_pdl(apply_kernel<80>, dim3(grid), dim3(128), 0, st_, X, sX, M, skk, out, sO, out_t, sT, ldt, R, up); break;
      case 96: err = launch_pdl(apply_kernel<96>, dim3(grid), dim3(128), 0, st_, X, sX, M, skk, out, sO, out_t, sT, ldt, R, up); break;
      default: err = cudaErrorInvalidValue; return;
    }
    err = cudaGetLastError();
  }

  // X [L][R][kp] <- orth(X) by rounds of shifted Cholesky QR (the first with
  // shift `first`, later ones kShiftSecond); tmp has X's shape.  With out_t
  // set, the last round writes bf16 X^T [kp][ldt] there instead of X.
  void orth(float*& X, float*& tmp, int64_t sX, int R, int k, int rounds, float first, float* g, float* rfac,
            uint16_t* out_t = nullptr, int64_t sT = 0, int ldt = 0) {
    for (int r = 0; r < rounds && err == cudaSuccess; ++r) {
      gram(X, sX, g, R);                                                      // G = X^T X
      chol(g, rfac, k, r == 0 ? first : kShiftSecond);                        // G + sI = R^T R
      if (r == rounds - 1 && out_t) {
        apply(X, sX, rfac, nullptr, 0, R, true, out_t, sT, ldt);              // (X R^-1)^T in bf16
      } else {
        apply(X, sX, rfac, tmp, sX, R, true);                                 // X R^-1
        std::swap(X, tmp);
      }
    }
  }

  size_t chol_smem() const { return 0; }   // chol_kernel's shared memory is static

  void chol(float* g, float* rfac, int k, float rel) {
    if (err != cudaSuccess) return;
    const int64_t skk = (int64_t)kp_ * kp_;
    switch (kp_) {
      case 16: err = launch_pdl(chol_kernel<16>, dim3(L_), dim3(kThreads), chol_smem(), st_, g, skk, rfac, skk, k, rel); break;
      case 32: err = launch_pdl(chol_kernel<32>, dim3(L_), dim3(kThreads), chol_smem(), st_, g, skk, rfac, skk, k, rel); break;
      case 48: err = launch_pdl(chol_kernel<48>, dim3(L_), dim3(kThreads), chol_smem(), st_, g, skk, rfac, skk, k, rel); break;
      case 64: err = launch_pdl(chol_kernel<64>, dim3(L_), dim3(kThreads), chol_smem(), st_, g, skk, rfac, skk, k, rel); break;
      case 80: err = launch_pdl(chol_kernel<80>, dim3(L_), dim3(kThreads), chol_smem(), st_, g, skk, rfac, skk, k, rel); break;
      case 96: err = launch_pdl(chol_kernel<96>, dim3(L_), dim3(kThreads), chol_smem(), st_, g, skk, rfac, skk, k, rel); break;
      default: err = cudaErrorInvalidValue; return;
    }
    err = cudaGetLastError();
  }
  size_t jacobi_smem() const { return sizeof(float) * ((size_t)(kp_ * (kp_ + 1) + 3) / 4 * 4 + (size_t)kp_ * (kp_ + 4)); }

  static cudaError_t configure() {
    cudaError_t e = cudaSuccess;
    const int jac = (int)(sizeof(float) * ((kMaxK * (kMaxK + 1) + 3) / 4 * 4 + kMaxK * (kMaxK + 4)));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(jacobi_kernel<kJacThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize, jac);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pass_smem_bytes(kMaxK));
    return e;
  }

 private:
  cudaStream_t st_;
  int L_, kp_, sms_;
  uint32_t* status_;
};

}  // namespace pf
}  // namespace kvrp

using namespace kvrp;

extern "C" {

size_t kv_patch_form_workspace_size(int32_t n_layers, int32_t n_tokens, int32_t row_width, int32_t rank,
                                    int32_t oversample) {
  if (n_layers <= 0 || n_tokens <= 0 || row_width <= 0 || rank <= 0 || oversample < 0) return 0;
  return pf::layout(nullptr, n_layers, n_tokens, row_width, pf::pad16(rank + oversample)).bytes + 1024;
}

kvrp_status kv_patch_form_orbit(const void* const* conditioned, const int64_t* deltas, int32_t n_orbit,
                                const void* canonical, int64_t cond_layer_stride, int64_t canon_layer_stride,
                                int32_t n_layers, int32_t n_tokens, int32_t row_width, int32_t rope_kind,
                                int32_t rot_dim, double rope_theta, int32_t rank, int32_t oversample,
                                int32_t power_iters, const float* omega, void* u_out, void* v_out,
                                int64_t u_layer_stride, int64_t v_layer_stride, void* workspace,
                                size_t workspace_bytes, uint32_t* d_status, kvrp_stream_t stream) {
  if (!conditioned || !deltas || !canonical || !omega || !u_out || !v_out)
    return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: NULL pointer argument");
  if (n_orbit <= 0 || n_orbit > pf::kMaxOrbit)
    return fail(KVRP_ERR_UNSUPPORTED, "kv_patch_form_orbit: 1 <= n_orbit <= %d", pf::kMaxOrbit);
  for (int p = 0; p < n_orbit; ++p) {
    if (!conditioned[p]) return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: conditioned cache %d is NULL", p);
    if (!aligned16(conditioned[p]))
      return fail(KVRP_ERR_ALIGNMENT, "kv_patch_form: conditioned cache %d is not 16-byte aligned", p);
  }
  if (!aligned16(canonical) || !aligned16(omega) || !aligned16(u_out) || !aligned16(v_out))
    return fail(KVRP_ERR_ALIGNMENT, "kv_patch_form: pointers must be 16-byte aligned");
  if (n_layers <= 0 || n_tokens <= 0 || row_width <= 0)
    return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: n_layers, n_tokens, row_width must be > 0");
  if (row_width % 4) return fail(KVRP_ERR_UNSUPPORTED, "kv_patch_form: row_width must be a multiple of 4");
  if (n_layers > 65535) return fail(KVRP_ERR_UNSUPPORTED, "kv_patch_form: at most 65535 layers");
  if (rope_kind != KVRP_ROPE_NONE && rope_kind != KVRP_ROPE_HEADS && rope_kind != KVRP_ROPE_MLA_TAIL)
    return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: unknown rope_kind %d", rope_kind);
  if (rope_kind != KVRP_ROPE_NONE) {
    if (rot_dim <= 0 || rot_dim % 4 || rot_dim > 2 * kTablePairs)
      return fail(KVRP_ERR_UNSUPPORTED, "kv_patch_form: rot_dim must be a multiple of 4 up to 128");
    if (rope_kind == KVRP_ROPE_HEADS && row_width % rot_dim)
      return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: row_width must be a multiple of rot_dim");
    if (rope_kind == KVRP_ROPE_MLA_TAIL && row_width <= rot_dim)
      return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: the rotated tail must fit the row");
    if (!(rope_theta > 0.0) || !std::isfinite(rope_theta))
      return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: rope_theta must be > 0");
  }
  const int k = rank + oversample;
  if (rank <= 0 || oversample < 0 || k > pf::kMaxK || rank > n_tokens || rank > row_width)
    return fail(KVRP_ERR_UNSUPPORTED, "kv_patch_form: need 0 < rank <= min(tokens, row), rank + oversample <= %d",
                pf::kMaxK);
  if (power_iters < 0 || power_iters > 8) return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: power_iters in 0..8");
  // a layer stride of 0 means dense layers
  if (cond_layer_stride == 0) cond_layer_stride = (int64_t)n_tokens * row_width;
  if (canon_layer_stride == 0) canon_layer_stride = (int64_t)n_tokens * row_width;
  if (u_layer_stride == 0) u_layer_stride = (int64_t)n_tokens * rank;
  if (v_layer_stride == 0) v_layer_stride = (int64_t)row_width * rank;
  if (n_layers > 1 && (cond_layer_stride < (int64_t)n_tokens * row_width ||
                       canon_layer_stride < (int64_t)n_tokens * row_width))
    return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: layer strides smaller than one layer");
  if (n_layers > 1 && (u_layer_stride < (int64_t)n_tokens * rank || v_layer_stride < (int64_t)row_width * rank))
    return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: factor layer strides smaller than one layer");
  if (cond_layer_stride % 2 || canon_layer_stride % 2)
    return fail(KVRP_ERR_ALIGNMENT, "kv_patch_form: cache layer strides must be even");
  const size_t need = kv_patch_form_workspace_size(n_layers, n_tokens, row_width, rank, oversample);
  if (!workspace || workspace_bytes < need)
    return fail(KVRP_ERR_WORKSPACE, "kv_patch_form: workspace of %zu bytes needed", need);
  int sms = 0, smem = 0;
  kvrp_status st0 = current_device_sms(&sms, &smem);
  if (st0 != KVRP_OK) return st0;
  cudaError_t e = pf::Runner::configure();
  if (e != cudaSuccess) return fail(KVRP_ERR_CUDA, "kv_patch_form: %s", cudaGetErrorString(e));
  if (!pf::encoder()) return fail(KVRP_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");

  cudaStream_t st = stream;
  const int L = n_layers, T = n_tokens, D = row_width, m = rank, kp = pf::pad16(k);
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(workspace) + 1023) & ~uintptr_t(1023));
  const pf::Buffers b = pf::layout(base, L, T, D, kp);

  // 1. Delta, rows and transposed rows, bf16
  pf::DeltaArgs da = {};
  for (int p = 0; p < n_orbit; ++p) da.cond[p] = static_cast<const uint16_t*>(conditioned[p]);
  da.canon = static_cast<const uint16_t*>(canonical);
  da.out = b.delta;
  da.out_t = b.delta_t;
  da.cond_stride = cond_layer_stride;
  da.canon_stride = canon_layer_stride;
  da.n_cond = n_orbit;
  da.T = T;
  da.D = D;
  da.Dp = (int)b.Dp;
  da.Tp = (int)b.Tp;
  da.rope_kind = rope_kind;
  da.rot_dim = rope_kind == KVRP_ROPE_NONE ? 4 : rot_dim;
  da.inv_n = 1.0f / (float)n_orbit;
  pf::TableParam tab = {};
  if (rope_kind != KVRP_ROPE_NONE) pf::mean_table(deltas, n_orbit, rope_theta, rot_dim, tab.v);
  da.g_zero = b.g;
  da.g_count = b.s_kk * L;
  e = pf::launch_pdl(pf::delta_kernel,
                     dim3((T + pf::kDeltaTokens - 1) / pf::kDeltaTokens, pf::segment_count(rope_kind, D, da.rot_dim), L),
                     dim3(pf::kThreads), 0, st, da, tab);
  if (e == cudaSuccess)
    e = pf::launch_pdl(pf::omega_t_kernel, dim3(std::max(1, std::min(sms, (D * kp + 255) / 256))), dim3(256), 0, st,
                       omega, D, k, b.omega_t, kp, (int)b.Dp);
  if (e != cudaSuccess) return fail(KVRP_ERR_CUDA, "kv_patch_form: %s", cudaGetErrorString(e));

  pf::Runner run(st, L, kp, sms, d_status);
  float *y = b.y, *y2 = b.y2, *z = b.z, *z2 = b.z2;
  // 2. range finder with subspace iterations (tensor-core passes over Delta and Delta^T)
  run.pass(b.delta, b.Dp, b.s_delta, b.omega_t, b.Dp, b.s_st_d, false, y, b.s_tk, T, D);           // Y = Delta Omega
  for (int it = 0; it < power_iters; ++it) {
    run.orth(y, y2, b.s_tk, T, k, 1, pf::kShiftFirst, b.g, b.rfac, b.st_t, b.s_st_t, (int)b.Tp);     // Q^T
    run.pass(b.delta_t, b.Tp, b.s_delta_t, b.st_t, b.Tp, b.s_st_t, true, z, b.s_dk, D, T);          // Z = Delta^T Q
    run.orth(z, z2, b.s_dk, D, k, 1, pf::kShiftFirst, b.g, b.rfac, b.st_d, b.s_st_d, (int)b.Dp);     // Zq^T
    run.pass(b.delta, b.Dp, b.s_delta, b.st_d, b.Dp, b.s_st_d, true, y, b.s_tk, T, D);              // Y = Delta Zq
  }
  // 3. Q = orth(Y); B^T = Delta^T Q; C = B B^T
  run.orth(y, y2, b.s_tk, T, k, 1, pf::kShiftFirst, b.g, b.rfac, b.st_t, b.s_st_t, (int)b.Tp);
  run.pass(b.delta_t, b.Tp, b.s_delta_t, b.st_t, b.Tp, b.s_st_t, true, z, b.s_dk, D, T);
  run.gram(z, b.s_dk, b.g, D);
  // 4. eigenvectors of the m largest eigenvalues, scaled by lambda^-1/2
  if (run.err == cudaSuccess && !run.map_fail) {
    run.err = pf::launch_pdl(pf::jacobi_kernel<pf::kJacThreads>, dim3(L), dim3(pf::kJacThreads), run.jacobi_smem(), st,
                             b.g, b.s_kk, b.w, b.s_kk, k, kp, m);
  }
  // 5. V_m = orth(B^T W) (columns already near unit length) as bf16 V^T; U_m = Delta V_m
  run.apply(z, b.s_dk, b.w, z2, b.s_dk, D, false);
  run.orth(z2, z, b.s_dk, D, m, 1, pf::kShiftSecond, b.g, b.rfac, b.st_d, b.s_st_d, (int)b.Dp);
  run.pass(b.delta, b.Dp, b.s_delta, b.st_d, b.Dp, b.s_st_d, true, y2, b.s_tk, T, D);
  if (run.err == cudaSuccess && !run.map_fail) {
    run.err = pf::launch_pdl(pf::u_out_kernel, dim3(64, L), dim3(256), 0, st, (const float*)y2, b.s_tk, kp,
                             static_cast<uint16_t*>(u_out), u_layer_stride, T, m);
    if (run.err == cudaSuccess)
      run.err = pf::launch_pdl(pf::v_out_kernel, dim3(64, L), dim3(256), 0, st, (const uint16_t*)b.st_d, b.s_st_d,
                               (int)b.Dp, static_cast<uint16_t*>(v_out), v_layer_stride, D, m);
  }
  if (run.map_fail) return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: cuTensorMapEncodeTiled rejected a workspace map");
  if (run.err != cudaSuccess) return fail(KVRP_ERR_CUDA, "kv_patch_form: %s", cudaGetErrorString(run.err));
  return KVRP_OK;
}

kvrp_status kv_patch_form(const void* conditioned, const void* canonical, int64_t cond_layer_stride,
                          int64_t canon_layer_stride, int32_t n_layers, int32_t n_tokens, int32_t row_width,
                          int32_t rope_kind, int32_t rot_dim, int64_t delta, double rope_theta, int32_t rank,
                          int32_t oversample, int32_t power_iters, const float* omega, void* u_out, void* v_out,
                          int64_t u_layer_stride, int64_t v_layer_stride, void* workspace, size_t workspace_bytes,
                          uint32_t* d_status, kvrp_stream_t stream) {
  const void* one[1] = {conditioned};
  return kv_patch_form_orbit(one, &delta, 1, canonical, cond_layer_stride, canon_layer_stride, n_layers, n_tokens,
                             row_width, rope_kind, rot_dim, rope_theta, rank, oversample, power_iters, omega, u_out,
                             v_out, u_layer_stride, v_layer_stride, workspace, workspace_bytes, d_status, stream);
}

}  // extern "C"
