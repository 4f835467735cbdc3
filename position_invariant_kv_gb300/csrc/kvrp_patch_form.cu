// Patch formation: the rank-m factors of the conditioning deficit.
//
// Kamera (gist.science/pt/paper/2606.23581, section 2, patch bullet) forms the
// patch once per chunk: a conditioned pass over [A, B] yields KV(B|A), and the
// top-m factors of the deficit come from an SVD.  Here the deficit is taken in
// the destination frame, Delta = KV(B|A) - R(delta) KV(B|empty), so that
// R(delta) KV(B|empty) + U_m V_m^T reproduces KV(B|A) up to the truncation.
// Singular values are folded into U_m, and the factors land in bf16 in the
// layout kv_relocate_patch reads.
//
// Method (all in this file's kernels, every layer of a call batched):
//   1. Delta in fp32 from the two bf16 caches (R(delta) with the split table);
//   2. randomized range finder: Y = Delta Omega (Omega: caller's Gaussian test
//      matrix), q power iterations Y <- Delta orth(Delta^T orth(Y));
//   3. Q = orth(Y) by two rounds of Cholesky QR (Gram in fp32, factor in fp64);
//   4. B = Q^T Delta and C = B B^T;
//   5. C = U_B Lambda U_B^T by parallel cyclic Jacobi in fp64 (one CTA);
//   6. V_m = B^T U_B[:, :m] with unit columns, U_m = Delta V_m (singular
//      values land in U_m).
// The tall products are tiled fp32 CUDA-core GEMMs: patch formation runs once
// per chunk, off the relocation hot path.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <vector>

#include "kvrp.h"
#include "kvrp_plan.h"

namespace kvrp {
namespace pf {

constexpr int kMaxK = 96;            // rank + oversampling bound (Jacobi works in shared memory)
constexpr int kJacobiSweeps = 20;
constexpr double kCholShift = 1e-6;  // Cholesky QR shift, relative to trace(G) (fp32 Gram)

struct TableParam {
  float4 v[kTablePairs];
};

// ---------------------------------------------------------------------------
// 1. Delta = conditioned - R(delta) canonical, fp32
// ---------------------------------------------------------------------------
struct DeltaArgs {
  const uint16_t* cond;
  const uint16_t* canon;
  int64_t cond_stride, canon_stride;   // elements between layers
  float* out;                          // layer l at out + l * out_stride, rows [T][D]
  int64_t out_stride;
  int T, D;
  int rope_kind;                       // KVRP_ROPE_*
  int rot_dim;                         // rotated head width (heads) or tail width (MLA)
};

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__global__ void __launch_bounds__(256) delta_kernel(DeltaArgs a, const __grid_constant__ TableParam tab) {
  const int t = blockIdx.x;
  const int l = blockIdx.y;
  const uint16_t* c = a.cond + (int64_t)l * a.cond_stride + (int64_t)t * a.D;
  const uint16_t* x = a.canon + (int64_t)l * a.canon_stride + (int64_t)t * a.D;
  float* o = a.out + (int64_t)l * a.out_stride + (int64_t)t * a.D;
  const int half = a.rot_dim / 2;
  const int rot_from = a.rope_kind == KVRP_ROPE_MLA_TAIL ? a.D - a.rot_dim : 0;
  for (int f = threadIdx.x; f < a.D / 2; f += blockDim.x) {
    // f indexes a pair of output elements (e0, e1) and, when they turn, the pair index i
    int e0, e1, i = -1;
    if (a.rope_kind == KVRP_ROPE_HEADS) {
      const int h = f / half;
      i = f % half;
      e0 = h * a.rot_dim + i;
      e1 = e0 + half;
    } else if (a.rope_kind == KVRP_ROPE_MLA_TAIL && 2 * f >= rot_from) {
      i = f - rot_from / 2;
      e0 = rot_from + i;
      e1 = e0 + half;
    } else {
      e0 = 2 * f;
      e1 = e0 + 1;
    }
    const float x0 = bf16f(x[e0]), x1 = bf16f(x[e1]);
    float y0 = x0, y1 = x1;
    if (i >= 0) {
      const float4 hd = tab.v[2 * (i >> 1)];
      const float4 tl = tab.v[2 * (i >> 1) + 1];
      const float C = (i & 1) ? hd.y : hd.x, S = (i & 1) ? hd.w : hd.z;
      const float Cl = (i & 1) ? tl.y : tl.x, Sl = (i & 1) ? tl.w : tl.z;
      y0 = fmaf(x0, C, -(x1 * S)) + fmaf(x0, Cl, -(x1 * Sl));
      y1 = fmaf(x1, C, x0 * S) + fmaf(x1, Cl, x0 * Sl);
    }
    o[e0] = bf16f(c[e0]) - y0;
    o[e1] = bf16f(c[e1]) - y1;
  }
}

// ---------------------------------------------------------------------------
// 2. Batched fp32 GEMM, C = op(A) op(B), 64 x 64 tiles, optional split-K
// ---------------------------------------------------------------------------
struct GemmArgs {
  const float* A;
  const float* B;
  float* C;
  int M, N, K;
  int lda, ldb, ldc;
  int64_t sA, sB, sC;   // batch strides (elements); 0 shares a matrix across the batch
  int tA, tB;           // A stored [K][M] / B stored [N][K]
  int splits;           // > 1: partial products are added into a zeroed C
};

__global__ void __launch_bounds__(256) gemm_f32(GemmArgs g) {
  const int z = blockIdx.z / g.splits;
  const int split = blockIdx.z % g.splits;
  const float* A = g.A + z * g.sA;
  const float* B = g.B + z * g.sB;
  float* C = g.C + z * g.sC;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int kchunk = ((g.K + g.splits - 1) / g.splits + 15) / 16 * 16;
  const int kb = split * kchunk;
  const int ke = min(g.K, kb + kchunk);
  __shared__ float As[16][68];
  __shared__ float Bs[16][68];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = kb; k0 < ke; k0 += 16) {
    for (int e = threadIdx.x; e < 1024; e += 256) {
      int mm, kk;
      if (g.tA) { mm = e & 63; kk = e >> 6; } else { kk = e & 15; mm = e >> 4; }
      const int gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < g.M && gk < ke) v = g.tA ? A[(int64_t)gk * g.lda + gm] : A[(int64_t)gm * g.lda + gk];
      As[kk][mm] = v;
      int nn, kk2;
      if (g.tB) { kk2 = e & 15; nn = e >> 4; } else { nn = e & 63; kk2 = e >> 6; }
      const int gn = n0 + nn, gk2 = k0 + kk2;
      float w = 0.f;
      if (gn < g.N && gk2 < ke) w = g.tB ? B[(int64_t)gn * g.ldb + gk2] : B[(int64_t)gk2 * g.ldb + gn];
      Bs[kk2][nn] = w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= g.N) continue;
      if (g.splits > 1) atomicAdd(&C[(int64_t)gm * g.ldc + gn], acc[i][j]);
      else C[(int64_t)gm * g.ldc + gn] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------
// 3. Cholesky QR step: from the Gram matrix G = X^T X (k x k), R^-1 with
//    G = R^T R (R upper), in fp64.  One CTA per batch entry.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) chol_inverse_kernel(const float* G, float* Rinv, int k) {
  extern __shared__ double sm[];
  double* R = sm;              // k x k
  double* X = sm + k * k;      // k x k
  __shared__ double shift;
  const float* g = G + (int64_t)blockIdx.x * k * k;
  float* out = Rinv + (int64_t)blockIdx.x * k * k;
  for (int e = threadIdx.x; e < k * k; e += blockDim.x) {
    const int i = e / k, j = e % k;
    R[e] = 0.5 * ((double)g[i * k + j] + (double)g[j * k + i]);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double tr = 0.0;
    for (int i = 0; i < k; ++i) tr += R[i * k + i];
    // Shifted Cholesky QR: G + s I with s well above the fp32 rounding of G keeps
    // the factorisation defined for a rank-deficient X; directions of X far
    // below sqrt(s) are damped instead of amplified, and the second round
    // restores orthonormality on the directions that carry signal.
    shift = tr > 0.0 ? kCholShift * tr : 1e-30;
  }
  __syncthreads();
  if (threadIdx.x < k) R[threadIdx.x * k + threadIdx.x] += shift;
  __syncthreads();
  // right-looking Cholesky, row j of R per step
  for (int j = 0; j < k; ++j) {
    if (threadIdx.x == 0) {
      double d = R[j * k + j];
      for (int i = 0; i < j; ++i) d -= R[i * k + j] * R[i * k + j];
      R[j * k + j] = sqrt(d > shift ? d : shift);
    }
    __syncthreads();
    for (int c = j + 1 + threadIdx.x; c < k; c += blockDim.x) {
      double v = R[j * k + c];
      for (int i = 0; i < j; ++i) v -= R[i * k + j] * R[i * k + c];
      R[j * k + c] = v / R[j * k + j];
    }
    __syncthreads();
  }
  // X = R^-1 (upper triangular), one column per thread, back substitution
  for (int c = threadIdx.x; c < k; c += blockDim.x) {
    for (int i = k - 1; i >= 0; --i) {
      double v = (i == c) ? 1.0 : 0.0;
      if (i > c) v = 0.0;
      else
        for (int j = i + 1; j <= c; ++j) v -= R[i * k + j] * X[j * k + c];
      X[i * k + c] = (i > c) ? 0.0 : v / R[i * k + i];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < k * k; e += blockDim.x) out[e] = (float)X[e];
}

// ---------------------------------------------------------------------------
// 5. Symmetric eigenproblem C = U L U^T by parallel cyclic Jacobi (round-robin
//    pairing: n/2 disjoint rotations per step), fp64, one CTA per entry.
//    Writes the eigenvectors of the m largest eigenvalues, W = U[:, top m]
//    (k x m, descending).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) jacobi_kernel(const float* Cm, float* W, int k, int m) {
  extern __shared__ double sm[];
  double* A = sm;                 // k x k
  double* V = sm + k * k;         // k x k
  __shared__ double cs_c[kMaxK / 2 + 1], cs_s[kMaxK / 2 + 1];
  __shared__ int pp[kMaxK / 2 + 1], qq[kMaxK / 2 + 1];
  __shared__ int idx[kMaxK + 1];
  __shared__ int order[kMaxK];
  __shared__ double red[256];
  __shared__ int done;
  __shared__ double floor_abs;
  const float* c = Cm + (int64_t)blockIdx.x * k * k;
  float* w = W + (int64_t)blockIdx.x * k * m;
  const int n2 = k + (k & 1);
  for (int e = threadIdx.x; e < k * k; e += blockDim.x) {
    const int i = e / k, j = e % k;
    A[e] = 0.5 * ((double)c[i * k + j] + (double)c[j * k + i]);
    V[e] = (i == j) ? 1.0 : 0.0;
  }
  for (int i = threadIdx.x; i < n2; i += blockDim.x) idx[i] = i;
  __syncthreads();
  {  // entries below 1e-15 ||C||_F are rounding noise of the fp32 input
    double ss = 0.0;
    for (int e = threadIdx.x; e < k * k; e += blockDim.x) ss += A[e] * A[e];
    red[threadIdx.x] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
      for (int i = 0; i < blockDim.x; ++i) t += red[i];
      floor_abs = 1e-15 * sqrt(t);
    }
    __syncthreads();
  }
  for (int sweep = 0; sweep < kJacobiSweeps; ++sweep) {
    // stop once every off-diagonal entry is negligible next to its diagonal pair
    double mx = 0.0;
    for (int e = threadIdx.x; e < k * k; e += blockDim.x) {
      const int i = e / k, j = e % k;
      if (i == j || fabs(A[e]) <= floor_abs) continue;
      const double r = fabs(A[e]) / sqrt(fabs(A[i * k + i] * A[j * k + j]) + 1e-300);
      mx = r > mx ? r : mx;
    }
    red[threadIdx.x] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
      double r = 0.0;
      for (int t = 0; t < blockDim.x; ++t) r = red[t] > r ? red[t] : r;
      done = r <= 1e-14;
    }
    __syncthreads();
    if (done) break;
    for (int step = 0; step < n2 - 1; ++step) {
      const int np = n2 / 2;
      if (threadIdx.x < np) {
        int p = idx[threadIdx.x], q = idx[n2 - 1 - threadIdx.x];
        if (p > q) { const int t = p; p = q; q = t; }
        double cc = 1.0, ss = 0.0;
        if (q < k) {
          const double apq = A[p * k + q];
          if (fabs(apq) > floor_abs && fabs(apq) > 1e-16 * sqrt(fabs(A[p * k + p] * A[q * k + q]))) {
            const double th = (A[q * k + q] - A[p * k + p]) / (2.0 * apq);
            const double t = fabs(th) < 1e150 ? ((th >= 0 ? 1.0 : -1.0) / (fabs(th) + sqrt(th * th + 1.0))) : 0.5 / th;
            cc = 1.0 / sqrt(t * t + 1.0);
            ss = t * cc;
          }
        }
        pp[threadIdx.x] = p;
        qq[threadIdx.x] = q;
        cs_c[threadIdx.x] = cc;
        cs_s[threadIdx.x] = ss;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < np * k; e += blockDim.x) {   // rows p, q
        const int t = e / k, j = e % k;
        const int p = pp[t], q = qq[t];
        if (q >= k) continue;
        const double cc = cs_c[t], ss = cs_s[t];
        const double ap = A[p * k + j], aq = A[q * k + j];
        A[p * k + j] = cc * ap - ss * aq;
        A[q * k + j] = ss * ap + cc * aq;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < np * k; e += blockDim.x) {   // columns p, q and eigenvectors
        const int t = e / k, j = e % k;
        const int p = pp[t], q = qq[t];
        if (q >= k) continue;
        const double cc = cs_c[t], ss = cs_s[t];
        const double ap = A[j * k + p], aq = A[j * k + q];
        A[j * k + p] = cc * ap - ss * aq;
        A[j * k + q] = ss * ap + cc * aq;
        const double vp = V[j * k + p], vq = V[j * k + q];
        V[j * k + p] = cc * vp - ss * vq;
        V[j * k + q] = ss * vp + cc * vq;
      }
      __syncthreads();
      if (threadIdx.x == 0) {   // next round of the tournament: keep idx[0], rotate the rest
        const int last = idx[n2 - 1];
        for (int i = n2 - 1; i > 1; --i) idx[i] = idx[i - 1];
        idx[1] = last;
      }
      __syncthreads();
    }
  }
  if (threadIdx.x == 0) {   // indices of the m largest eigenvalues, descending
    for (int j = 0; j < k; ++j) order[j] = j;
    for (int a = 0; a < m; ++a) {
      int best = a;
      for (int b = a + 1; b < k; ++b)
        if (A[order[b] * k + order[b]] > A[order[best] * k + order[best]]) best = b;
      const int t = order[a]; order[a] = order[best]; order[best] = t;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < k * m; e += blockDim.x) {
    const int i = e / m, j = e % m;
    w[i * m + j] = (float)V[i * k + order[j]];
  }
}

// ---------------------------------------------------------------------------
// 6a. V_m = B^T U_B has columns of norm sqrt(lambda_j); scale each to unit
//     length from its own computed norm (not from lambda, whose fp32 rounding
//     can be far off for a vanishing eigenvalue).  A zero column stays zero.
//     One CTA per layer.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) normalise_columns_kernel(float* Vm, int64_t stride, int rows, int m) {
  __shared__ double part[256];
  __shared__ float scale[kMaxK];
  float* v = Vm + (int64_t)blockIdx.x * stride;
  for (int j = 0; j < m; ++j) {
    double ss = 0.0;
    for (int r = threadIdx.x; r < rows; r += blockDim.x) ss += (double)v[(int64_t)r * m + j] * v[(int64_t)r * m + j];
    part[threadIdx.x] = ss;
    __syncthreads();
    for (int h = blockDim.x / 2; h > 0; h >>= 1) {
      if (threadIdx.x < h) part[threadIdx.x] += part[threadIdx.x + h];
      __syncthreads();
    }
    if (threadIdx.x == 0) scale[j] = part[0] > 0.0 ? (float)(1.0 / sqrt(part[0])) : 0.f;
    __syncthreads();
  }
  for (int64_t e = threadIdx.x; e < (int64_t)rows * m; e += blockDim.x) v[e] *= scale[e % m];
}

// ---------------------------------------------------------------------------
// 6. fp32 -> bf16 factors in the caller's layout
// ---------------------------------------------------------------------------
__global__ void to_bf16_kernel(const float* src, int64_t src_stride, uint16_t* dst, int64_t dst_stride,
                               int64_t n_per_layer) {
  const int l = blockIdx.y;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n_per_layer;
       e += (int64_t)gridDim.x * blockDim.x) {
    const __nv_bfloat16 b = __float2bfloat16_rn(src[l * src_stride + e]);
    dst[l * dst_stride + e] = *reinterpret_cast<const uint16_t*>(&b);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct Buffers {
  float *delta, *y, *y2, *z, *z2, *b, *g, *rinv, *c, *w, *vf, *uf;
  int64_t s_delta, s_tk, s_dk, s_kd, s_kk, s_km, s_dm, s_tm;
  size_t bytes;
};

size_t round64(size_t v) { return (v + 63) / 64 * 64; }

Buffers layout(float* base, int L, int T, int D, int k, int m) {
  Buffers b;
  b.s_delta = (int64_t)round64((size_t)T * D);
  b.s_tk = (int64_t)round64((size_t)T * k);
  b.s_dk = (int64_t)round64((size_t)D * k);
  b.s_kd = (int64_t)round64((size_t)k * D);
  b.s_kk = (int64_t)round64((size_t)k * k);
  b.s_km = (int64_t)round64((size_t)k * m);
  b.s_dm = (int64_t)round64((size_t)D * m);
  b.s_tm = (int64_t)round64((size_t)T * m);
  float* p = base;
  auto take = [&](int64_t stride) {
    float* q = p;
    p += stride * L;
    return q;
  };
  b.delta = take(b.s_delta);
  b.y = take(b.s_tk);
  b.y2 = take(b.s_tk);
  b.z = take(b.s_dk);
  b.z2 = take(b.s_dk);
  b.b = take(b.s_kd);
  b.g = take(b.s_kk);
  b.rinv = take(b.s_kk);
  b.c = take(b.s_kk);
  b.w = take(b.s_km);
  b.vf = take(b.s_dm);
  b.uf = take(b.s_tm);
  b.bytes = (size_t)(p - base) * sizeof(float);
  return b;
}

cudaError_t gemm(cudaStream_t st, int L, const float* A, int64_t sA, int lda, int tA, const float* B, int64_t sB,
                 int ldb, int tB, float* C, int64_t sC, int ldc, int M, int N, int K, int splits) {
  GemmArgs g{A, B, C, M, N, K, lda, ldb, ldc, sA, sB, sC, tA, tB, splits};
  if (splits > 1) {
    for (int l = 0; l < L; ++l) {   // split-K partials are added into zeros
      const cudaError_t e = cudaMemsetAsync(C + l * sC, 0, sizeof(float) * (size_t)M * ldc, st);
      if (e != cudaSuccess) return e;
    }
  }
  dim3 grid((N + 63) / 64, (M + 63) / 64, L * splits);
  gemm_f32<<<grid, 256, 0, st>>>(g);
  return cudaGetLastError();
}

int splits_for(int K) { return K >= 2048 ? 16 : K >= 512 ? 4 : 1; }

// X [rows x k] (batched) <- X R^-1, twice (Cholesky QR2); tmp is a buffer of X's shape.
cudaError_t orthonormalise(cudaStream_t st, int L, float* X, float* tmp, int64_t sX, int rows, int k, float* g,
                           float* rinv, int64_t s_kk) {
  for (int round = 0; round < 2; ++round) {
    cudaError_t e = gemm(st, L, X, sX, k, 1, X, sX, k, 0, g, s_kk, k, k, k, rows, splits_for(rows));
    if (e != cudaSuccess) return e;
    chol_inverse_kernel<<<L, 256, 2 * sizeof(double) * k * k, st>>>(g, rinv, k);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = gemm(st, L, X, sX, k, 0, rinv, s_kk, k, 0, tmp, sX, k, rows, k, k, 1);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyAsync(X, tmp, sizeof(float) * (size_t)sX * L, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pf
}  // namespace kvrp

using namespace kvrp;

extern "C" {

size_t kv_patch_form_workspace_size(int32_t n_layers, int32_t n_tokens, int32_t row_width, int32_t rank,
                                    int32_t oversample) {
  if (n_layers <= 0 || n_tokens <= 0 || row_width <= 0 || rank <= 0 || oversample < 0) return 0;
  const int k = rank + oversample;
  return pf::layout(nullptr, n_layers, n_tokens, row_width, k, rank).bytes + 256;
}

kvrp_status kv_patch_form(const void* conditioned, const void* canonical, int64_t cond_layer_stride,
                          int64_t canon_layer_stride, int32_t n_layers, int32_t n_tokens, int32_t row_width,
                          int32_t rope_kind, int32_t rot_dim, int64_t delta, double rope_theta, int32_t rank,
                          int32_t oversample, int32_t power_iters, const float* omega, void* u_out, void* v_out,
                          int64_t u_layer_stride, int64_t v_layer_stride, void* workspace, size_t workspace_bytes,
                          kvrp_stream_t stream) {
  if (!conditioned || !canonical || !omega || !u_out || !v_out)
    return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: NULL pointer argument");
  if (!aligned16(conditioned) || !aligned16(canonical) || !aligned16(omega) || !aligned16(u_out) ||
      !aligned16(v_out))
    return fail(KVRP_ERR_ALIGNMENT, "kv_patch_form: pointers must be 16-byte aligned");
  if (n_layers <= 0 || n_tokens <= 0 || row_width <= 0 || row_width % 2)
    return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: n_layers, n_tokens > 0 and an even row_width are required");
  if (rope_kind != KVRP_ROPE_NONE && rope_kind != KVRP_ROPE_HEADS && rope_kind != KVRP_ROPE_MLA_TAIL)
    return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: unknown rope_kind %d", rope_kind);
  if (rope_kind != KVRP_ROPE_NONE) {
    if (rot_dim <= 0 || rot_dim % 4 || rot_dim > 2 * kTablePairs)
      return fail(KVRP_ERR_UNSUPPORTED, "kv_patch_form: rot_dim must be a multiple of 4 up to 128");
    if (rope_kind == KVRP_ROPE_HEADS && row_width % rot_dim)
      return fail(KVRP_ERR_INVALID_ARG, "kv_patch_form: row_width must be a multiple of rot_dim");
    if (rope_kind == KVRP_ROPE_MLA_TAIL && (row_width <= rot_dim || (row_width - rot_dim) % 2))
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
  const size_t need = kv_patch_form_workspace_size(n_layers, n_tokens, row_width, rank, oversample);
  if (!workspace || workspace_bytes < need)
    return fail(KVRP_ERR_WORKSPACE, "kv_patch_form: workspace of %zu bytes needed", need);
  int sms = 0, smem = 0;
  kvrp_status st0 = current_device_sms(&sms, &smem);
  if (st0 != KVRP_OK) return st0;

  cudaStream_t st = stream;
  const int L = n_layers, T = n_tokens, D = row_width, m = rank;
  float* base = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255));
  const pf::Buffers b = pf::layout(base, L, T, D, k, m);
  pf::TableParam tab = {};
  const int64_t d3[3] = {delta, 0, 0};
  const int32_t s3[3] = {rot_dim / 2, 0, 0};
  if (rope_kind != KVRP_ROPE_NONE) phase_table(d3, s3, rope_theta, rot_dim, tab.v);

  cudaError_t e = cudaSuccess;
  // the kernels of steps 3 and 5 keep k x k fp64 matrices in shared memory
  e = cudaFuncSetAttribute(pf::chol_inverse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           2 * (int)sizeof(double) * pf::kMaxK * pf::kMaxK);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pf::jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             2 * (int)sizeof(double) * pf::kMaxK * pf::kMaxK);
  if (e != cudaSuccess) return fail(KVRP_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  // Gram-type matrices are used densely (leading dimension k)
  const int64_t s_kk = (int64_t)k * k;
  float* g = b.g;
  float* rinv = b.rinv;
  float* cmat = b.c;

  // 1. Delta
  pf::DeltaArgs da{static_cast<const uint16_t*>(conditioned), static_cast<const uint16_t*>(canonical),
                   cond_layer_stride, canon_layer_stride, b.delta, b.s_delta, T, D, rope_kind, rot_dim};
  pf::delta_kernel<<<dim3(T, L), 256, 0, st>>>(da, tab);
  e = cudaGetLastError();
  // 2. range finder with power iterations
  if (e == cudaSuccess) e = pf::gemm(st, L, b.delta, b.s_delta, D, 0, omega, 0, k, 0, b.y, b.s_tk, k, T, k, D, 1);
  for (int it = 0; it < power_iters && e == cudaSuccess; ++it) {
    e = pf::orthonormalise(st, L, b.y, b.y2, b.s_tk, T, k, g, rinv, s_kk);
    if (e == cudaSuccess)
      e = pf::gemm(st, L, b.delta, b.s_delta, D, 1, b.y, b.s_tk, k, 0, b.z, b.s_dk, k, D, k, T, pf::splits_for(T));
    if (e == cudaSuccess) e = pf::orthonormalise(st, L, b.z, b.z2, b.s_dk, D, k, g, rinv, s_kk);
    if (e == cudaSuccess) e = pf::gemm(st, L, b.delta, b.s_delta, D, 0, b.z, b.s_dk, k, 0, b.y, b.s_tk, k, T, k, D, 1);
  }
  // 3. Q = orth(Y)
  if (e == cudaSuccess) e = pf::orthonormalise(st, L, b.y, b.y2, b.s_tk, T, k, g, rinv, s_kk);
  // 4. B = Q^T Delta  (k x D), C = B B^T  (k x k)
  if (e == cudaSuccess)
    e = pf::gemm(st, L, b.y, b.s_tk, k, 1, b.delta, b.s_delta, D, 0, b.b, b.s_kd, D, k, D, T, pf::splits_for(T));
  if (e == cudaSuccess) e = pf::gemm(st, L, b.b, b.s_kd, D, 0, b.b, b.s_kd, D, 1, cmat, s_kk, k, k, k, D, pf::splits_for(D));
  // 5. eigenvectors of the m largest eigenvalues, W = U_B[:, :m]
  if (e == cudaSuccess) {
    pf::jacobi_kernel<<<L, 256, 2 * sizeof(double) * k * k, st>>>(cmat, b.w, k, m);
    e = cudaGetLastError();
  }
  // 6. V_m = B^T W normalised (D x m), U_m = Delta V_m (T x m)
  if (e == cudaSuccess) e = pf::gemm(st, L, b.b, b.s_kd, D, 1, b.w, (int64_t)k * m, m, 0, b.vf, b.s_dm, m, D, m, k, 1);
  if (e == cudaSuccess) {
    pf::normalise_columns_kernel<<<L, 256, 0, st>>>(b.vf, b.s_dm, D, m);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = pf::gemm(st, L, b.delta, b.s_delta, D, 0, b.vf, b.s_dm, m, 0, b.uf, b.s_tm, m, T, m, D, 1);
  if (e == cudaSuccess) {
    pf::to_bf16_kernel<<<dim3(64, L), 256, 0, st>>>(b.uf, b.s_tm, static_cast<uint16_t*>(u_out),
                                                    u_layer_stride, (int64_t)T * m);
    pf::to_bf16_kernel<<<dim3(64, L), 256, 0, st>>>(b.vf, b.s_dm, static_cast<uint16_t*>(v_out),
                                                    v_layer_stride, (int64_t)D * m);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return fail(KVRP_ERR_CUDA, "kv_patch_form: %s", cudaGetErrorString(e));
  return KVRP_OK;
}

}  // extern "C"
