// Relocation + rank-m patch kernel for GB300 (sm_103a).
//
// Computes, for every token row of every (chunk, tensor, layer) in a plan,
//     out = RN_bf16( R(delta) x + U_m V_m^T )
// and writes the row into its 16-token destination page (Kamera,
// gist.science/pt/paper/2606.23581, section 2 "O Operador Kamera": relocation
// by an exact RoPE re-rotation, then the rank-m conditioning patch).
//
// One persistent CTA per SM walks a list of items.  An item is a 128-token
// tile of one (chunk, tensor, layer), split into 128-feature sub-tiles.
// Warp roles:
//   warp 0      TMA producer: U tile per item, X sub-tile + V_m slice per stage
//   warp 1      TMEM owner and tcgen05.mma issuer: P = U V_m^T into TMEM (fp32)
//   warps 2..9  epilogue: one token row per thread, R(delta) in fp32 registers
//               with a split (16-bit head + fp32 tail) phase table, + P from
//               TMEM, round to bf16 in place in shared memory; then TMA stores
//               of whole destination pages and plain stores for edge rows.
// X and the destination pages move through 128B-swizzled shared memory, so the
// row-per-thread epilogue reads and writes without bank conflicts.
// Every wait is bounded; a stuck pipeline sets KVRP_DEV_TIMEOUT and the CTA
// drains its copies, frees its TMEM and returns.
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "kvrp.h"
#include "kvrp_plan.h"
#include "kvrp_ptx.h"

namespace kvrp {

struct alignas(64) ParamPlan {
  unsigned char bytes[kParamPlanBytes];
};

namespace dev {

using namespace kvrp::ptx;   // mbarrier, TMA, tcgen05 wrappers

// Two TMEM reads of N consecutive fp32 columns each (this warp's 32 lanes),
// completed (tcgen05.wait::ld) inside the same asm statement.
#define KVRP_R8(a, o) "=r"(a[o + 0]), "=r"(a[o + 1]), "=r"(a[o + 2]), "=r"(a[o + 3]), \
                      "=r"(a[o + 4]), "=r"(a[o + 5]), "=r"(a[o + 6]), "=r"(a[o + 7])
__device__ __forceinline__ void tmem_ld_2x16(uint32_t ta, uint32_t tb, uint32_t (&a)[16],
                                             uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : KVRP_R8(a, 0), KVRP_R8(a, 8), KVRP_R8(b, 0), KVRP_R8(b, 8)
      : "r"(ta), "r"(tb)
      : "memory");
}
#undef KVRP_R8

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
// No "memory" clobber: the shared-memory loads and stores of the epilogue are
// volatile asm, so they keep their order among themselves, while ordinary
// loads (the phase table) may be scheduled across them.  The proxy fence that
// precedes every TMA store carries the clobber.
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w));
}
__device__ __forceinline__ void stg128(void* p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Shared-memory matrix descriptor: K-major operand staged by a 32-byte
// swizzled TMA box (rows of 16 bf16 = 32 B, 8-row atoms 256 B apart).
__device__ __forceinline__ uint64_t desc_k_sw32(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused: K fits the atom)
  d |= (uint64_t)(256 >> 4) << 32;             // stride byte offset: next 8-row atom
  d |= (uint64_t)1 << 46;                      // descriptor version (tcgen05)
  d |= (uint64_t)6 << 61;                      // layout: 32-byte swizzle
  return d;
}
// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major, M = 128.
__device__ __forceinline__ uint32_t idesc_bf16_f32(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// --------------------------------------------------------------------------
// Plan access
// --------------------------------------------------------------------------
struct Item {
  const ChunkRec* c;
  const TensorRec* t;
  int tensor, layer, tblk, s0, s1;
  int t0;          // token index of tile row 0 (may be negative)
  int64_t q0;      // destination position of tile row 0
};

__device__ __forceinline__ Item decode_item(const unsigned char* plan, const PlanHdr& h, int item) {
  Item it;
  it.tensor = item >= h.items0 ? 1 : 0;
  const int local = item - (it.tensor ? h.items0 : 0);
  const int sg = local % h.n_sg;
  const int rest = local / h.n_sg;
  const int tiles = it.tensor ? h.tiles[1] : h.tiles[0];   // a select keeps the header in registers
  const int tile = rest % tiles;
  it.layer = rest / tiles;
  // the chunk holding this tile: last prefix-sum entry <= tile
  const int32_t* tbeg = reinterpret_cast<const int32_t*>(plan + h.off_tbeg) + it.tensor * (h.n_chunks + 1);
  int lo = 0, hi = h.n_chunks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tbeg[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  it.c = reinterpret_cast<const ChunkRec*>(plan + h.off_chunks) + lo;
  it.t = &it.c->t[it.tensor];
  it.tblk = tile - tbeg[lo];
  it.s0 = sg * h.subs_per_item;
  it.s1 = min(it.s0 + h.subs_per_item, h.n_sub);
  const int lead = (int)(it.t->dst_start % kPage);
  it.t0 = it.tblk * kTileRows - lead;
  it.q0 = it.t->dst_start - lead + (int64_t)it.tblk * kTileRows;
  return it;
}

__device__ __forceinline__ const CUtensorMap* plan_map(const unsigned char* plan, const PlanHdr& h,
                                                       int idx) {
  return reinterpret_cast<const CUtensorMap*>(plan + h.off_maps) + idx;
}

// --------------------------------------------------------------------------
// Epilogue arithmetic on one thread's share of a sub-tile row
// --------------------------------------------------------------------------
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Address of 16-byte chunk k (0..15) of tile row r inside a 128B-swizzled X sub-tile.
__device__ __forceinline__ uint32_t x_chunk_addr(uint32_t xbase, int r, int k) {
  return xbase + ((uint32_t)(k >> 3) << 14) + ((uint32_t)r << 7) + ((uint32_t)((k & 7) ^ (r & 7)) << 4);
}

// Rotate two neighbouring pairs at once with packed fp32x2 arithmetic.  xl /
// xh hold the lower / upper elements of pairs (i, i+1); `head` holds their
// 16-significant-bit cos and sin heads {C_i, C_i+1, S_i, S_i+1}, `tail` the
// fp32 remainders {Cl_i, Cl_i+1, Sl_i, Sl_i+1}.  Because a bf16 value times a
// 16-bit head is exact in fp32, x_l*C - x_h*S is formed with one rounding;
// the tails add the rest of the fp64 cos/sin.  Every packed operation rounds
// each lane exactly like its scalar counterpart.
__device__ __forceinline__ float2 neg2(float2 v) { return make_float2(-v.x, -v.y); }

__device__ __forceinline__ void turn2(float2 xl, float2 xh, float4 head, float4 tail, float2& yl,
                                      float2& yh) {
  const float2 C = make_float2(head.x, head.y), S = make_float2(head.z, head.w);
  const float2 Cl = make_float2(tail.x, tail.y), Sl = make_float2(tail.z, tail.w);
  const float2 b = __ffma2_rn(xl, C, neg2(__fmul2_rn(xh, S)));
  const float2 tl = __ffma2_rn(xl, Cl, neg2(__fmul2_rn(xh, Sl)));
  const float2 b2 = __ffma2_rn(xh, C, __fmul2_rn(xl, S));
  const float2 th = __ffma2_rn(xh, Cl, __fmul2_rn(xl, Sl));
  yl = __fadd2_rn(b, tl);
  yh = __fadd2_rn(b2, th);
}
__device__ __forceinline__ void turn2_patch(float2 xl, float2 xh, float4 head, float4 tail, float2 pl,
                                            float2 ph, float2& yl, float2& yh) {
  const float2 C = make_float2(head.x, head.y), S = make_float2(head.z, head.w);
  const float2 Cl = make_float2(tail.x, tail.y), Sl = make_float2(tail.z, tail.w);
  const float2 b = __ffma2_rn(xl, C, neg2(__fmul2_rn(xh, S)));
  const float2 tl = __ffma2_rn(xl, Cl, neg2(__fmul2_rn(xh, Sl)));
  const float2 b2 = __ffma2_rn(xh, C, __fmul2_rn(xl, S));
  const float2 th = __ffma2_rn(xh, Cl, __fmul2_rn(xl, Sl));
  yl = __fadd2_rn(b, __fadd2_rn(tl, pl));
  yh = __fadd2_rn(b2, __fadd2_rn(th, ph));
}

// N = columns per part (32 or 16).  The thread owns two parts of N columns
// starting at a0 and a1; with ROT, element j of part a pairs with element j
// of part b and uses table entry tab0 + j.  Accumulators are read in rounds of
// 16 columns per part to keep register use low.
template <int N, bool ROT, bool PATCH>
__device__ __forceinline__ void epilogue_part(uint32_t xbase, int row, int a0, int a1, const float4* tab, int tab0,
                                              uint32_t tm_a, uint32_t tm_b) {
#pragma unroll
  for (int r0 = 0; r0 < N; r0 += 16) {
    uint32_t pa[16], pb[16];
    if constexpr (PATCH) tmem_ld_2x16(tm_a + r0, tm_b + r0, pa, pb);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t addr_a = x_chunk_addr(xbase, row, ((a0 + r0) >> 3) + k);
      const uint32_t addr_b = x_chunk_addr(xbase, row, ((a1 + r0) >> 3) + k);
      const uint4 va = lds128(addr_a);
      const uint4 vb = lds128(addr_b);
      const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
      const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
      uint32_t oa[4], ob[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int e = 8 * k + 2 * w;        // elements e, e + 1 of both parts
        const float2 xl = make_float2(bf_lo(wa[w]), bf_hi(wa[w]));
        const float2 xh = make_float2(bf_lo(wb[w]), bf_hi(wb[w]));
        float2 yl, yh;
        if constexpr (ROT) {
          // table entries are stored two pairs at a time; all lanes read the same
          // entry (a broadcast), from shared or global memory through one pointer
          const float4 head = tab[tab0 + r0 + e];
          const float4 tail = tab[tab0 + r0 + e + 1];
          if constexpr (PATCH) {
            turn2_patch(xl, xh, head, tail, make_float2(__uint_as_float(pa[e]), __uint_as_float(pa[e + 1])),
                        make_float2(__uint_as_float(pb[e]), __uint_as_float(pb[e + 1])), yl, yh);
          } else {
            turn2(xl, xh, head, tail, yl, yh);
          }
        } else {
          yl = __fadd2_rn(xl, make_float2(__uint_as_float(pa[e]), __uint_as_float(pa[e + 1])));
          yh = __fadd2_rn(xh, make_float2(__uint_as_float(pb[e]), __uint_as_float(pb[e + 1])));
        }
        oa[w] = pack_bf2(yl.x, yl.y);
        ob[w] = pack_bf2(yh.x, yh.y);
      }
      sts128(addr_a, make_uint4(oa[0], oa[1], oa[2], oa[3]));
      sts128(addr_b, make_uint4(ob[0], ob[1], ob[2], ob[3]));
    }
  }
}

// --------------------------------------------------------------------------
// The kernel
// --------------------------------------------------------------------------
// mbarriers: per shared-memory stage (X sub-tile + V_m slice) full/empty,
// per TMEM accumulator slot full/empty, per U buffer full/empty, and one
// drain barrier for the MMA issuer's last commit.
struct Bars {
  uint32_t base;
  __device__ uint32_t full(int s) const { return base + 8u * s; }
  __device__ uint32_t empty(int s) const { return base + 8u * (kMaxStages + s); }
  __device__ uint32_t acc_full(int a) const { return base + 8u * (2 * kMaxStages + a); }
  __device__ uint32_t acc_empty(int a) const { return base + 8u * (2 * kMaxStages + kAccSlots + a); }
  __device__ uint32_t u_full(int b) const { return base + 8u * (2 * kMaxStages + 2 * kAccSlots + b); }
  __device__ uint32_t u_empty(int b) const { return base + 8u * (2 * kMaxStages + 2 * kAccSlots + 2 + b); }
  __device__ uint32_t drain() const { return base + 8u * (2 * kMaxStages + 2 * kAccSlots + 4); }
  __device__ uint32_t computed(int s) const { return base + 8u * (2 * kMaxStages + 2 * kAccSlots + 5 + s); }
};
static_assert(8 * (3 * kMaxStages + 2 * kAccSlots + 5) <= 512, "barriers must fit below the TMEM slot");

template <bool kParamPlan>
__global__ void __launch_bounds__(kThreads, 1)
    relocate_kernel(const __grid_constant__ ParamPlan pp, const unsigned char* __restrict__ gplan) {
  const unsigned char* plan = kParamPlan ? pp.bytes : gplan;
  const PlanHdr h = *reinterpret_cast<const PlanHdr*>(plan);

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const SmemLayout L = smem_layout(h.m_max, h.stages, h.u_bufs, h.tab_mode);
  const uint32_t NU = (uint32_t)h.u_bufs;
  const uint32_t sbase = smem_u32(smem);
  const Bars bars{sbase};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 520);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = h.stages;
  // limit of the pipeline waits below (the drains at the end keep the default:
  // a copy or MMA in flight always completes, and must, before the CTA exits)
  const long long wlim = h.wait_cycles ? (long long)h.wait_cycles : kTimeoutCycles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bars.full(s), 1);
      // released by the owning group's store warp and, when there is an MMA issuer, by it
      mbar_init(bars.empty(s), 1 + (h.tmem_cols > 0 ? 1 : 0));
      mbar_init(bars.computed(s), kGroupWarps);   // the group's rows are final in shared memory
    }
    for (int a = 0; a < kAccSlots; ++a) {
      mbar_init(bars.acc_full(a), 1);
      mbar_init(bars.acc_empty(a), kGroupWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.u_full(b), 1);
      mbar_init(bars.u_empty(b), 1);
    }
    mbar_init(bars.drain(), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1 && h.tmem_cols > 0) tmem_alloc(smem_u32(tmem_slot), (uint32_t)h.tmem_cols);
  if (h.tab_mode == kTabFixed && h.n_tables == 1 && threadIdx.x < kTablePairs) {
    // a plan with one phase table keeps it in shared memory for the whole launch
    const float4 v = reinterpret_cast<const float4*>(plan + h.off_tabs)[threadIdx.x];
    reinterpret_cast<float4*>(smem + L.tab_off)[threadIdx.x] = v;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = h.tmem_cols > 0 ? *tmem_slot : 0u;
  // Programmatic dependent launch: the set-up above may overlap the previous
  // kernel on this stream; nothing global is touched before it has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const uint32_t u_buf0 = sbase + L.u_off;
  auto u_buf = [&](int b) { return u_buf0 + (uint32_t)b * L.u_bytes; };
  auto x_buf = [&](int s) { return sbase + L.stage_off + (uint32_t)s * L.stage_bytes; };
  auto w_buf = [&](int s) { return x_buf(s) + L.x_bytes; };
  // shared-memory table slot of a stage (kTabStaged), or the fixed copy (kTabFixed)
  auto tab_buf = [&](int s) { return sbase + L.tab_off + (h.tab_mode == kTabStaged ? (uint32_t)s * kTableBytes : 0u); };
  const float4* tab_smem = reinterpret_cast<const float4*>(smem + L.tab_off);
  const float4* tab_glob = reinterpret_cast<const float4*>(plan + h.off_tabs);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t it = 0, uit = 0;
      bool ok = true;
      // A plan in global memory was written by an earlier kernel: before this
      // thread's first TMA use of each tensor map it acquires the map through
      // the tensor-map proxy (maps in the parameter block need no fence).
      int32_t acq_x = -1, acq_u = -1, acq_w = -1;
      for (int item = blockIdx.x; ok && item < h.n_items; item += gridDim.x) {
        const Item I = decode_item(plan, h, item);
        const int m = I.c->rank;
        const int nkb = (m + 15) >> 4;          // 16-rank MMA steps; a rank-8 tail box reads zeros
        if (!kParamPlan) {
          if (I.t->map_x != acq_x) tensormap_acquire(plan_map(plan, h, acq_x = I.t->map_x));
          if (m > 0 && I.t->map_u != acq_u) tensormap_acquire(plan_map(plan, h, acq_u = I.t->map_u));
          if (m > 0 && I.t->map_w != acq_w) tensormap_acquire(plan_map(plan, h, acq_w = I.t->map_w));
        }
        if (h.tab_mode == kTabGlobal && item + (int)gridDim.x < h.n_items) {
          // warm L1 with the next item's phase table for the epilogue
          const Item N = decode_item(plan, h, item + (int)gridDim.x);
          if (N.c->table >= 0 && N.t->rot_kind != kRotNone) {
            const unsigned char* tp = plan + h.off_tabs + (size_t)N.c->table * kTableBytes;
            for (int l = 0; l < kTableBytes; l += 128) prefetch_l1(tp + l);
          }
        }
        if (m > 0) {
          const int ub = (int)(uit % NU);
          ok = wait_phase(bars.u_empty(ub), ((uit / NU) & 1) ^ 1, abort_flag, h.status, wlim);
          if (!ok) break;
          const CUtensorMap* mu = plan_map(plan, h, I.t->map_u);
          mbar_expect_tx(bars.u_full(ub), (uint32_t)nkb * (kTileRows * 32));
          for (int k = 0; k < nkb; ++k)
            tma_load_3d(u_buf(ub) + (uint32_t)k * (kTileRows * 32), mu, bars.u_full(ub), 16 * k, I.t0,
                        I.layer);
          ++uit;
        }
        const CUtensorMap* mx = plan_map(plan, h, I.t->map_x);
        const CUtensorMap* mw = m > 0 ? plan_map(plan, h, I.t->map_w) : nullptr;
        for (int s = I.s0; s < I.s1; ++s, ++it) {
          const int st = (int)(it % (uint32_t)S);
          ok = wait_phase(bars.empty(st), ((it / S) & 1) ^ 1, abort_flag, h.status, wlim);
          if (!ok) break;
          const int width = min(kSubCols, h.D - kSubCols * s);
          const int nbox = width / kBoxCols;
          uint32_t bytes = (uint32_t)nbox * (kTileRows * kBoxCols * 2);
          if (m > 0) bytes += (uint32_t)nkb * (uint32_t)width * 32u;
          const bool copy_tab = h.tab_mode == kTabStaged && I.t->rot_kind != kRotNone;
          if (copy_tab) bytes += kTableBytes;
          mbar_expect_tx(bars.full(st), bytes);
          if (copy_tab)
            bulk_load(tab_buf(st), plan + h.off_tabs + (size_t)I.c->table * kTableBytes, kTableBytes,
                      bars.full(st));
          for (int j = 0; j < nbox; ++j)
            tma_load_3d(x_buf(st) + (uint32_t)j * (kTileRows * kBoxCols * 2), mx, bars.full(st),
                        kSubCols * s + kBoxCols * j, I.t->x_row0 + I.t0, I.layer);
          for (int k = 0; k < nkb; ++k)
            for (int j = 0; j < nbox; ++j)
              tma_load_3d(w_buf(st) + (uint32_t)k * (uint32_t)width * 32u + (uint32_t)j * (kBoxCols * 32),
                          mw, bars.full(st), 16 * k, kSubCols * s + kBoxCols * j, I.layer);
        }
      }
      // Let every copy this CTA started land before the CTA can exit.
      const uint32_t first = it > (uint32_t)S ? it - (uint32_t)S : 0u;
      for (uint32_t j = first; j < it; ++j) {
        volatile int no_abort = 0;
        wait_phase(bars.full((int)(j % (uint32_t)S)), (j / S) & 1, &no_abort, nullptr);
      }
      const uint32_t ufirst = uit > NU ? uit - NU : 0u;
      for (uint32_t j = ufirst; j < uit; ++j) {
        volatile int no_abort = 0;
        wait_phase(bars.u_full((int)(j % NU)), (j / NU) & 1, &no_abort, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && h.tmem_cols > 0) {
      uint32_t it = 0, uit = 0;
      uint32_t gcnt[kEpiGroups] = {};   // patched sub-tiles issued into each group's slot
      bool ok = true;
      bool issued = false;
      for (int item = blockIdx.x; ok && item < h.n_items; item += gridDim.x) {
        const Item I = decode_item(plan, h, item);
        const int m = I.c->rank;
        const int nkb = (m + 15) >> 4;
        const int ub = (int)(uit % NU);
        if (m > 0) {
          ok = wait_phase(bars.u_full(ub), (uit / NU) & 1, abort_flag, h.status, wlim);
          if (!ok) break;
        }
        for (int s = I.s0; s < I.s1; ++s, ++it) {
          const int st = (int)(it % (uint32_t)S);
          // observe every stage use, patched or not, and take part in its release
          ok = wait_phase(bars.full(st), (it / S) & 1, abort_flag, h.status, wlim);
          if (!ok) break;
          if (m > 0) {
            const int a = (int)(it % kEpiGroups);     // the slot of the group that owns this stage
            ok = wait_phase(bars.acc_empty(a), (gcnt[a] & 1) ^ 1, abort_flag, h.status, wlim);
            if (!ok) break;
            tc_fence_after();
            const int width = min(kSubCols, h.D - kSubCols * s);
            const uint32_t idesc = idesc_bf16_f32(width);
            const uint32_t d_tmem = tmem_base + (uint32_t)a * kSubCols;
            for (int k = 0; k < nkb; ++k) {
              const uint64_t ad = desc_k_sw32(u_buf(ub) + (uint32_t)k * (kTileRows * 32));
              const uint64_t bd = desc_k_sw32(w_buf(st) + (uint32_t)k * (uint32_t)width * 32u);
              mma_bf16(d_tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
            }
            mma_commit(bars.acc_full(a));
            issued = true;
            ++gcnt[a];
          }
          // the group releases the stage only after acc_full, i.e. after these MMAs read it
          mbar_arrive(bars.empty(st));
        }
        if (!ok) break;
        if (m > 0) {
          mma_commit(bars.u_empty(ub));
          ++uit;
        }
      }
      if (issued) {
        // every MMA this thread issued has completed once `drain` flips
        mma_commit(bars.drain());
        volatile int no_abort = 0;
        wait_phase(bars.drain(), 0, &no_abort, nullptr);
      }
    }
  } else if (warp >= 2 + kEpilogueWarps) {
    // ------------------------------------------------------------ page stores
    // One warp per epilogue group.  When the group's rows of a stage are final
    // it stores every whole 16-row page of the tile by TMA (lane p: page p),
    // waits until those stores have read shared memory, and releases the stage.
    const int group = warp - 2 - kEpilogueWarps;
    uint32_t it = 0;
    bool ok = true;
    int32_t acq_dst = -1;                    // last destination map this lane acquired (see the producer)
    for (int item = blockIdx.x; ok && item < h.n_items; item += gridDim.x) {
      const Item I = decode_item(plan, h, item);
      const TensorRec& T = *I.t;
      const CUtensorMap* md = plan_map(plan, h, T.map_dst);
      if (!kParamPlan && T.map_dst != acq_dst) tensormap_acquire(plan_map(plan, h, acq_dst = T.map_dst));
      const int r_lo = max(0, -I.t0);
      const int r_hi = min(kTileRows, I.c->n_tokens - I.t0);
      const int p = lane;                                   // page of the tile this lane stores
      const bool whole = p < kTileRows / kPage && kPage * p >= r_lo && kPage * p + kPage <= r_hi;
      int64_t page = -1;
      if (whole) {
        const int64_t lp = (I.q0 + kPage * p) / kPage;
        page = T.block_table ? (int64_t)__ldg(T.block_table + lp) : lp;
      }
      for (int s = I.s0; s < I.s1; ++s, ++it) {
        if ((int)(it % kEpiGroups) != group) continue;   // another group's sub-tile
        const int st = (int)(it % (uint32_t)S);
        ok = wait_phase(bars.computed(st), (it / S) & 1, abort_flag, h.status, wlim);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (whole) {
          if (page < 0 || page >= T.num_pages) {
            if (h.status) atomicOr(h.status, KVRP_DEV_BAD_PAGE);
          } else {
            const int width = min(kSubCols, h.D - kSubCols * s);
            const uint32_t xb = x_buf(st);
            for (int j = 0; j < width / kBoxCols; ++j)
              tma_store_3d(md, xb + (uint32_t)j * (kTileRows * kBoxCols * 2) + (uint32_t)p * (kPage * 128u),
                           kSubCols * s + kBoxCols * j, (int)(page * kPage), I.layer);
            bulk_commit();
            bulk_wait_read_0();
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.empty(st));
      }
    }
    bulk_wait_0();   // this warp's page stores are complete before the CTA exits
  } else {
    // --------------------------------------------------------------- epilogue
    // Two groups of four warps take sub-tiles in turn (group g owns the stages
    // s with s % 2 == g, so it sees every phase of them).  Each warp owns the
    // 32 tile rows of its TMEM lane quarter across all columns, so it needs no
    // other warp: it turns, patches and rounds its rows in shared memory, then
    // lanes 0 and 16 store the warp's two 16-row pages by TMA.
    const int ew = warp - 2;                 // 0..7
    const int group = ew / kGroupWarps;      // which sub-tiles this warp serves
    const int quarter = warp & 3;            // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;     // tile row (token) of this thread
    uint32_t it = 0;
    uint32_t gait = 0;                       // patched sub-tiles this group has taken
    const uint32_t tslot = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)group * kSubCols;
    bool aborted = false;
    for (int item = blockIdx.x; !aborted && item < h.n_items; item += gridDim.x) {
      const Item I = decode_item(plan, h, item);
      const int m = I.c->rank;
      const TensorRec& T = *I.t;
      const int n_tok = I.c->n_tokens;
      // valid tile rows [r_lo, r_hi); this thread's row and its destination page
      const int r_lo = max(0, -I.t0);
      const int r_hi = min(kTileRows, n_tok - I.t0);
      const bool valid = row >= r_lo && row < r_hi;
      const int pg_row = row & ~(kPage - 1);
      const bool whole_page = pg_row >= r_lo && pg_row + kPage <= r_hi;
      int64_t page = -1;
      if (valid) {
        const int64_t lp = (I.q0 + row) / kPage;
        page = T.block_table ? (int64_t)__ldg(T.block_table + lp) : lp;   // used at store time
      }
      for (int s = I.s0; s < I.s1; ++s, ++it) {
        if ((int)(it % kEpiGroups) != group) continue;   // another group's sub-tile
        const int st = (int)(it % (uint32_t)S);
        bool ok = wait_phase(bars.full(st), (it / S) & 1, abort_flag, h.status, wlim);
        if (ok && m > 0) {
          ok = wait_phase(bars.acc_full(group), gait & 1, abort_flag, h.status, wlim);
          tc_fence_after();
        }
        ok = __all_sync(0xffffffffu, ok);     // TMEM loads below are warp-collective
        if (!ok) {
          aborted = true;
          break;
        }
        const int width = min(kSubCols, h.D - kSubCols * s);
        const uint32_t xb = x_buf(st);
        const float4* tab = h.tab_mode == kTabGlobal
                                ? (I.c->table >= 0 ? tab_glob + (size_t)I.c->table * kTablePairs : tab_glob)
                                : tab_smem + (h.tab_mode == kTabStaged ? st * kTablePairs : 0);
        const uint32_t tcol = tslot;
        if (width == kSubCols && T.rot_kind == kRotHalf128) {
          // one head of 128: column j pairs with j + 64
          if (m > 0) epilogue_part<64, true, true>(xb, row, 0, 64, tab, 0, tcol, tcol + 64);
          else epilogue_part<64, true, false>(xb, row, 0, 64, tab, 0, 0, 0);
        } else {
          // each 64-wide box on its own: turned (pairs j, j + 32) or not
          for (int b = 0; b < width / kBoxCols; ++b) {
            const int a0 = kBoxCols * b;
            const bool rot = T.rot_kind == kRotHalf64 && kSubCols * s + a0 >= T.rot_from;
            if (m > 0) {
              if (rot) epilogue_part<32, true, true>(xb, row, a0, a0 + 32, tab, 0, tcol + a0, tcol + a0 + 32);
              else epilogue_part<32, false, true>(xb, row, a0, a0 + 32, tab, 0, tcol + a0, tcol + a0 + 32);
            } else if (rot) {
              epilogue_part<32, true, false>(xb, row, a0, a0 + 32, tab, 0, 0, 0);
            }
          }
        }
        if (m > 0) {
          // release this accumulator slot to the MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.acc_empty(group));
          ++gait;
        }
        fence_proxy_async_smem();
        __syncwarp();

        // ---- rows of partly covered pages go out now, by their own threads;
        //      whole pages are left to the group's store warp
        if (valid && !whole_page) {
          if (page < 0 || page >= T.num_pages) {
            if (h.status) atomicOr(h.status, KVRP_DEV_BAD_PAGE);
          } else {
            uint16_t* dst_row = T.dst + (int64_t)I.layer * T.dst_layer_stride +
                                (page * kPage + (I.q0 + row) % kPage) * (int64_t)h.D + kSubCols * s;
            for (int c = 0; c < width / 8; ++c) stg128(dst_row + 8 * c, lds128(x_chunk_addr(xb, row, c)));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.computed(st));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1 && h.tmem_cols > 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)h.tmem_cols);
  }
}

}  // namespace dev

// ---------------------------------------------------------------------------
// Allocation-free batch path.  The launch plan of kv_relocate_batch_noalloc
// lives in this fixed device array instead of a caller-provided workspace, so
// that callers who cannot allocate device memory can still run a batch.  Every
// GPU that loads the library holds the array until the process exits; all
// calls on a device share it.
// ---------------------------------------------------------------------------
namespace {
// Sized for the largest plan a batch of KVRP_NOALLOC_MAX_CHUNKS chunks can
// produce (the same bound kv_relocate_batch_workspace_size reports).
static __device__ __align__(256) unsigned char g_noalloc_plan[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
std::map<int, void*> g_noalloc_ptr;   // device ordinal -> device address of g_noalloc_plan
}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

cudaError_t noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  auto found = g_noalloc_ptr.find(dev);
  if (found != g_noalloc_ptr.end()) {
    *ptr = found->second;
    return cudaSuccess;
  }
  // In host code g_noalloc_plan names a host-side stand-in, not device
  // memory: the device address must come from the runtime, per device, with
  // that device current.
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_plan);
  if (e != cudaSuccess) return e;
  g_noalloc_ptr[dev] = p;
  *ptr = p;
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// Plan upload.  A batch plan is carried to device memory in the parameter
// blocks of small copy kernels (up to 31 KB each): the launch copies the bytes
// when it is enqueued, so the host plan may be freed as soon as the call
// returns, and no pinned staging buffer is needed.
// ---------------------------------------------------------------------------
namespace dev {
constexpr uint32_t kPieceBytes = 31 * 1024;
struct alignas(16) PlanPiece {
  unsigned char bytes[kPieceBytes];
};
// The parameter block is read through the constant cache, which serves the
// distinct addresses of a warp one after another; spreading a piece over
// several CTAs (SMs) reads it in parallel.
constexpr int kCopyCtas = 16, kCopyThreads = 128;
static_assert(kCopyCtas * kCopyThreads * 16 >= (int)kPieceBytes, "one 16-byte word per thread");
__global__ void __launch_bounds__(kCopyThreads) plan_copy_kernel(const __grid_constant__ PlanPiece piece,
                                                                  unsigned char* __restrict__ dst, uint32_t n_bytes) {
  const uint32_t i = (blockIdx.x * kCopyThreads + threadIdx.x) * 16u;
  if (i < n_bytes) *reinterpret_cast<uint4*>(dst + i) = *reinterpret_cast<const uint4*>(piece.bytes + i);
}
}  // namespace dev

cudaError_t upload_plan(const void* host_bytes, size_t n_bytes, void* dev_plan, cudaStream_t stream) {
  if (n_bytes % 16 != 0) return cudaErrorInvalidValue;
  const unsigned char* src = static_cast<const unsigned char*>(host_bytes);
  unsigned char* dst = static_cast<unsigned char*>(dev_plan);
  dev::PlanPiece* piece = new dev::PlanPiece;   // 31 KB: off the stack
  cudaError_t e = cudaSuccess;
  for (size_t off = 0; off < n_bytes && e == cudaSuccess; off += dev::kPieceBytes) {
    const uint32_t n = (uint32_t)std::min<size_t>(dev::kPieceBytes, n_bytes - off);
    memcpy(piece->bytes, src + off, n);
    const int ctas = (int)((n + 16u * dev::kCopyThreads - 1) / (16u * dev::kCopyThreads));
    dev::plan_copy_kernel<<<ctas, dev::kCopyThreads, 0, stream>>>(*piece, dst + off, n);
    e = cudaGetLastError();
  }
  delete piece;
  return e;
}

int32_t upload_launches(size_t n_bytes) { return (int32_t)((n_bytes + dev::kPieceBytes - 1) / dev::kPieceBytes); }

cudaError_t prepare_kernel(int smem_bytes) {
  cudaError_t e = cudaFuncSetAttribute(dev::relocate_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(dev::relocate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem_bytes);
}

cudaError_t launch_relocate(const void* param_plan, const void* dev_plan, int grid, int smem_bytes,
                            cudaStream_t stream) {
  ParamPlan pp;
  if (param_plan) {
    // Single-chunk plans travel in the parameter block; such a launch may start
    // its set-up while the previous kernel on the stream drains.
    memcpy(pp.bytes, param_plan, kParamPlanBytes);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const unsigned char* none = nullptr;
    return cudaLaunchKernelEx(&cfg, dev::relocate_kernel<true>, pp, none);
  } else {
    dev::relocate_kernel<false><<<grid, kThreads, smem_bytes, stream>>>(
        pp, static_cast<const unsigned char*>(dev_plan));
  }
  return cudaGetLastError();
}

}  // namespace kvrp
