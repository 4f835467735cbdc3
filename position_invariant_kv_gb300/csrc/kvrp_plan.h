// Launch plan shared by the host side (kvrp_host.cpp) and the kernel
// (kvrp_kernel.cu).  A plan is one byte blob: a header, the TMA tensor maps,
// the per-chunk phase tables, the chunk records and per-tensor tile prefix sums.
// Small plans (one chunk) travel as a __grid_constant__ kernel parameter;
// batch plans are copied into a caller-provided device workspace.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvrp.h"

namespace kvrp {

constexpr int kPage = 16;           // tokens per destination page
constexpr int kTileRows = 128;      // tokens per tile (TMEM lanes / MMA M)
constexpr int kSubCols = 128;       // features per sub-tile (MMA N)
constexpr int kBoxCols = 64;        // features per 128-byte swizzled TMA box
constexpr int kMaxRank = 128;
constexpr int kTablePairs = 64;     // phase-table entries (head_dim / 2 <= 64)
constexpr int kParamPlanBytes = 3072;
constexpr int kGroupWarps = 4;      // epilogue warps that share one sub-tile (one per TMEM lane quarter)
constexpr int kEpiGroups = 2;       // epilogue groups, taking sub-tiles in turn
constexpr int kEpilogueWarps = kGroupWarps * kEpiGroups;
// Every mbarrier waiter must see each phase it waits on in order, or a phase
// two uses old could pass for the current one.  Hence: stage s belongs to
// epilogue group s % kEpiGroups (the depth is a multiple of kEpiGroups), each
// group owns one TMEM accumulator slot, and the MMA issuer observes every
// stage use (its arrival is part of the stage's release).
constexpr int kAccSlots = kEpiGroups;
// Pipeline depth bound.  Measured on GB300: 4 stages (2 per group) beat 6 by
// about 4% on unpatched work, whose deeper carve-out leaves less L1 for the
// phase-table and plan loads; patched work fits at most 4 anyway.
constexpr int kMaxStages = 4;
// warps: producer, MMA issuer, epilogue groups, then one page-store warp per group
constexpr int kThreads = 64 + 32 * kEpilogueWarps + 32 * kEpiGroups;

// Rotation kinds of one tensor.
enum RotKind : int32_t {
  kRotNone = 0,     // values, MLA at rank 0 ... : nothing turns
  kRotHalf128 = 1,  // heads of 128: feature i pairs with i + 64 inside each sub-tile
  kRotHalf64 = 2,   // heads of 64 (or MLA k_rope): i pairs with i + 32 inside each
                    // 64-wide box whose first feature is >= rot_from
};

struct TensorRec {             // one (chunk, tensor)
  int32_t map_x, map_u, map_w, map_dst;   // plan map indices; -1 when unused
  const int32_t* block_table;             // NULL = contiguous destination
  uint16_t* dst;                          // pool base (bf16 bits)
  int64_t dst_layer_stride;               // elements
  int64_t dst_start;
  int32_t num_pages;
  int32_t rot_kind;
  int32_t rot_from;                       // first rotated feature (kRotHalf64)
  int32_t n_tblk;                         // token tiles of this tensor
  int32_t x_row0;                         // row of the chunk's token 0 in its source map (see below)
  int32_t pad_;
};
// Source maps: chunks whose canonical rows follow one another in memory (same
// layer stride, each starting where the previous one ends) share one tensor
// map over all their rows, and a chunk addresses its rows from x_row0.  Tile
// rows outside the chunk then read its neighbours' rows (or the map's zero
// fill at the group's ends); they are loaded but never stored.

struct ChunkRec {
  TensorRec t[2];
  int32_t n_tokens;
  int32_t rank;
  int32_t n_tensors;
  int32_t table;                          // phase-table index; -1 when no tensor turns
};

struct PlanHdr {
  int32_t n_chunks;
  int32_t n_items;
  int32_t D;                              // row width (features)
  int32_t n_layers;
  int32_t n_sub;                          // sub-tiles per row: ceil(D / 128)
  int32_t subs_per_item;
  int32_t n_sg;                           // sub-tile groups per tile
  int32_t stages;                         // pipeline depth
  int32_t m_max;                          // largest rank in the plan (multiple of 16)
  int32_t tmem_cols;                      // allocated TMEM columns (0 = none)
  int32_t u_bufs;                         // U tile buffers (2, or 1 at the largest ranks)
  int32_t n_tables;                       // distinct phase tables in the plan
  int32_t tab_mode;                       // where the epilogue reads tables: kTab* below
  int32_t n_tensors;                      // tensors per chunk (GQA/MHA: K and V; MLA: 1)
  int32_t tiles[2];                       // token tiles over all chunks, per tensor
  int32_t items0;                         // items of tensor 0 (all layers)
  // Items run tensor-major, then layer, then chunk, then tile, then sub-tile
  // group: CTAs working side by side stream neighbouring chunks of one layer.
  uint32_t off_maps, off_tabs, off_chunks, off_tbeg;   // off_tbeg: int32 [n_tensors][n_chunks + 1] tile prefix sums
  uint32_t total_bytes;
  uint32_t wait_cycles;                   // pipeline wait limit in cycles; 0 = the default (~1 s)
  uint32_t* status;                       // optional device status word
};
static_assert(sizeof(PlanHdr) <= 128, "header must fit in 128 bytes");

// Upper bound of a serialised plan for n chunks of up to two tensors: header,
// up to 8 tensor maps and one phase table per chunk, the chunk records and the
// per-tensor tile prefix sums (n + 1 entries for each of two tensors).
constexpr size_t plan_align(size_t v) { return (v + 127) & ~static_cast<size_t>(127); }
constexpr size_t plan_bytes_bound(int64_t n) {
  return plan_align(plan_align(plan_align(plan_align(plan_align(sizeof(PlanHdr)) +
                                                     (size_t)n * 8 * sizeof(CUtensorMap)) +
                                          (size_t)n * kTablePairs * 16) +
                               (size_t)n * sizeof(ChunkRec)) +
                    (size_t)2 * (size_t)(n + 1) * sizeof(int32_t));
}

// Shared-memory carve-up for a given rank bound and depth.
constexpr int kTableBytes = kTablePairs * 16;   // one phase table: 64 float4

// Where the epilogue reads phase tables from.
enum TabMode : int32_t {
  kTabFixed = 0,     // the plan's only table, copied to shared memory once per launch
  kTabStaged = 1,    // one table per pipeline stage, copied with the stage's data
  kTabGlobal = 2,    // read from the plan in global memory; the producer prefetches
                     // the next item's table into L1 (when shared memory is full)
};

struct SmemLayout {
  uint32_t u_off, u_bytes;        // U buffers
  uint32_t stage_off, stage_bytes;
  uint32_t x_bytes, w_bytes;      // inside a stage: X sub-tile, then W slice
  uint32_t tab_off;               // phase-table slots (see TabMode)
  uint32_t total;
};

__host__ __device__ inline SmemLayout smem_layout(int m_max, int stages, int u_bufs, int tab_mode) {
  SmemLayout s;
  const uint32_t kb = (uint32_t)(m_max / 16);
  s.u_off = 1024;                                  // barriers live in the first 1 KB
  s.u_bytes = kb * (kTileRows * 32);               // one U buffer
  s.x_bytes = kTileRows * kSubCols * 2;            // 32 KB
  s.w_bytes = kb * (kSubCols * 32);
  s.stage_bytes = s.x_bytes + s.w_bytes;
  s.stage_off = s.u_off + (uint32_t)u_bufs * s.u_bytes;
  s.tab_off = s.stage_off + (uint32_t)stages * s.stage_bytes;
  const uint32_t n_tab = tab_mode == kTabFixed ? 1u : tab_mode == kTabStaged ? (uint32_t)stages : 0u;
  s.total = s.tab_off + n_tab * kTableBytes;
  return s;
}

// Launches the relocation kernel.  Exactly one of param_plan / dev_plan is used:
// param_plan (host bytes, <= kParamPlanBytes) travels as a kernel parameter,
// dev_plan points at a plan already resident in device memory.
cudaError_t launch_relocate(const void* param_plan, const void* dev_plan, int grid,
                            int smem_bytes, cudaStream_t stream);

// Copies a serialised plan (host bytes, a multiple of 16) to device memory on
// `stream` by small copy kernels whose parameter blocks carry the bytes, so no
// host buffer has to outlive the call and nothing is staged or pinned.
cudaError_t upload_plan(const void* host_bytes, size_t n_bytes, void* dev_plan, cudaStream_t stream);
// Copy launches upload_plan makes for a plan of n_bytes.
int32_t upload_launches(size_t n_bytes);

// Host helpers shared by the library's translation units.
kvrp_status fail(kvrp_status st, const char* fmt, ...);
// Kernel launches of this host thread's last relocation or attention call.
extern thread_local int32_t g_last_launches;
bool aligned16(const void* p);
// Split phase table of one shift: sections = frequency pairs per (t, h, w)
// section (plain RoPE: {rot_dim / 2, 0, 0}); layout as the kernel reads it.
void phase_table(const int64_t delta[3], const int32_t sections[3], double theta, int rot_dim, float4* tab);
// SM count and shared-memory opt-in limit of the current device (checks sm_103).
kvrp_status current_device_sms(int* sms, int* smem_optin);

// Per-device one-time kernel setup (dynamic shared-memory opt-in).
cudaError_t prepare_kernel(int smem_bytes);

// Allocation-free batch path: the largest batch its fixed device array holds,
// the array's size, and its device address on the current device (looked up
// once per device with cudaGetSymbolAddress).
constexpr int kNoAllocMaxChunks = KVRP_NOALLOC_MAX_CHUNKS;
constexpr size_t kNoAllocScratchBytes = plan_bytes_bound(kNoAllocMaxChunks);
size_t noalloc_scratch_bytes();
cudaError_t noalloc_scratch(void** ptr);

// Wait limit (cycles) written into every relocation plan; 0 keeps the default.
// Set only through kvrp_test_set_wait_limit, by tests of the failure path.
uint32_t test_wait_limit();

}  // namespace kvrp
