// Host side of libkvrp: argument checks, per-chunk phase tables, TMA tensor
// maps, the launch plan, and the three public entry points of kvrp.h.
//
// Operator: Kamera, gist.science/pt/paper/2606.23581, section 2 "O Operador
// Kamera" (KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T; GQA/MHA/MLA bullets)
// and section 3 (reorder, sliding-window survival and recall as many chunks
// with their own delta and patch, served here by kv_relocate_batch).
#include <cudaTypedefs.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "kvrp.h"
#include "kvrp_plan.h"

namespace kvrp {

thread_local char g_last_error[512] = "";
thread_local int32_t g_last_launches = 0;

kvrp_status fail(kvrp_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

kvrp_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVRP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

namespace {

// ---------------------------------------------------------------------------
// Per-device state: SM count, shared-memory limit, driver entry point.
// ---------------------------------------------------------------------------
struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
  int prepared_smem = 0;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_dev;
std::atomic<uint32_t> g_test_wait_limit{0};   // kvrp_test_set_wait_limit
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

kvrp_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return fail(KVRP_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  DeviceInfo& d = g_dev[dev];
  if (d.sms == 0) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(smem)");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) {
      d.sms = 0;
      return fail(KVRP_ERR_UNSUPPORTED, "libkvrp is built for sm_103a; device %d is sm_%d%d", dev, major,
                  minor);
    }
  }
  *out = &d;
  return KVRP_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// Phase tables: phi_i = delta * theta^(-2i/d) in fp64; cos and sin split into a
// 16-significant-bit head (so that a bf16 times the head is exact in fp32) and
// an fp32 tail holding the rest of the fp64 value.
// ---------------------------------------------------------------------------
float head16(double v) {
  if (v == 0.0) return 0.0f;
  int e = 0;
  const double m = std::frexp(v, &e);
  return static_cast<float>(std::ldexp(std::nearbyint(std::ldexp(m, 16)), e - 16));
}

// Layout, two pairs per float4 so the kernel can use packed fp32x2 math:
//   tab[2j]     = {C_2j,  C_2j+1,  S_2j,  S_2j+1}    (16-bit heads)
//   tab[2j + 1] = {Cl_2j, Cl_2j+1, Sl_2j, Sl_2j+1}   (fp32 tails)
// Frequency pair i turns by the shift of the section that holds it: plain
// RoPE has one section covering every pair; M-RoPE (multimodal RoPE of
// Qwen-VL-style models) has consecutive temporal / height / width sections.
void phase_table(const int64_t delta[3], const int32_t sections[3], double theta, int rot_dim, float4* tab) {
  float head_c[kTablePairs] = {}, head_s[kTablePairs] = {}, tail_c[kTablePairs] = {}, tail_s[kTablePairs] = {};
  int sec = 0, sec_end = sections[0];
  for (int i = 0; i < rot_dim / 2; ++i) {
    while (i >= sec_end && sec < 2) sec_end += sections[++sec];
    const double inv = std::pow(theta, -2.0 * i / rot_dim);
    const double phi = static_cast<double>(delta[sec]) * inv;
    const double c = std::cos(phi), s = std::sin(phi);
    head_c[i] = head16(c);
    head_s[i] = head16(s);
    tail_c[i] = static_cast<float>(c - head_c[i]);
    tail_s[i] = static_cast<float>(s - head_s[i]);
  }
  for (int j = 0; j < kTablePairs / 2; ++j) {
    tab[2 * j] = make_float4(head_c[2 * j], head_c[2 * j + 1], head_s[2 * j], head_s[2 * j + 1]);
    tab[2 * j + 1] = make_float4(tail_c[2 * j], tail_c[2 * j + 1], tail_s[2 * j], tail_s[2 * j + 1]);
  }
}

namespace {

// ---------------------------------------------------------------------------
// Chunk descriptions common to every entry point.
// ---------------------------------------------------------------------------
struct TensorIn {
  const void* src;
  const void* u;
  const void* w;
  kvrp_dst dst;
  int rot_kind;
  int rot_from;
};
struct ChunkIn {
  TensorIn t[2];
  int n_tensors;
  int64_t src_layer_stride, u_layer_stride, w_layer_stride;
  int32_t n_tokens, rank;
  int64_t delta[3];           // plain RoPE: {delta, 0, 0}
  int32_t sections[3];        // frequency pairs per section; plain RoPE: {rot_dim / 2, 0, 0}
};
struct Shape {
  int n_layers;
  int D;
  int rot_dim;   // 0 when nothing turns
  double theta;
};

kvrp_status check_dst(const kvrp_dst* d, const char* name, int64_t n_tokens, const Shape& sh) {
  if (!d) return fail(KVRP_ERR_INVALID_ARG, "%s is NULL", name);
  if (!d->base) return fail(KVRP_ERR_INVALID_ARG, "%s.base is NULL", name);
  if (!aligned16(d->base)) return fail(KVRP_ERR_ALIGNMENT, "%s.base is not 16-byte aligned", name);
  if (d->page_size != kPage) return fail(KVRP_ERR_UNSUPPORTED, "%s.page_size must be 16", name);
  if (d->num_pages <= 0 || (int64_t)d->num_pages * kPage > (1ll << 31) - 1)
    return fail(KVRP_ERR_INVALID_ARG, "%s.num_pages out of range", name);
  if (d->dst_start < 0) return fail(KVRP_ERR_INVALID_ARG, "%s.dst_start is negative", name);
  const int64_t pool = (int64_t)d->num_pages * kPage * sh.D;
  if (sh.n_layers > 1 && d->layer_stride < pool)
    return fail(KVRP_ERR_INVALID_ARG, "%s.layer_stride smaller than one layer's pool", name);
  if (d->layer_stride % 8 != 0) return fail(KVRP_ERR_ALIGNMENT, "%s.layer_stride not a multiple of 8", name);
  if (d->block_table) {
    if (reinterpret_cast<uintptr_t>(d->block_table) & 3u)
      return fail(KVRP_ERR_ALIGNMENT, "%s.block_table is not 4-byte aligned", name);
  } else if (d->dst_start + n_tokens > (int64_t)d->num_pages * kPage) {
    return fail(KVRP_ERR_INVALID_ARG, "%s: contiguous destination too small for the chunk", name);
  }
  return KVRP_OK;
}

kvrp_status check_chunk(const ChunkIn& c, const Shape& sh) {
  if (c.n_tokens < 0) return fail(KVRP_ERR_INVALID_ARG, "n_tokens is negative");
  if (c.rank < 0 || c.rank > kMaxRank || c.rank % 8 != 0)
    return fail(KVRP_ERR_UNSUPPORTED, "rank must be 0 or a multiple of 8 up to %d (got %d)", kMaxRank, c.rank);
  if (c.n_tokens > (1 << 30)) return fail(KVRP_ERR_INVALID_ARG, "n_tokens too large");
  const int64_t rows = c.n_tokens;
  if (sh.n_layers > 1 && c.src_layer_stride < rows * sh.D)
    return fail(KVRP_ERR_INVALID_ARG, "src_layer_stride smaller than one layer of rows");
  if (c.src_layer_stride % 8 != 0) return fail(KVRP_ERR_ALIGNMENT, "src_layer_stride not a multiple of 8");
  if (c.rank > 0) {
    if (sh.n_layers > 1 && c.u_layer_stride < rows * c.rank)
      return fail(KVRP_ERR_INVALID_ARG, "u_layer_stride smaller than one layer of U_m");
    if (sh.n_layers > 1 && c.w_layer_stride < (int64_t)sh.D * c.rank)
      return fail(KVRP_ERR_INVALID_ARG, "v_layer_stride smaller than one layer of V_m");
    if (c.u_layer_stride % 8 != 0 || c.w_layer_stride % 8 != 0)
      return fail(KVRP_ERR_ALIGNMENT, "factor layer strides must be multiples of 8");
  }
  static const char* names[2][3] = {{"k source", "K patch U_m", "K patch V_m"},
                                    {"v source", "V patch U_m", "V patch V_m"}};
  for (int t = 0; t < c.n_tensors; ++t) {
    const TensorIn& ti = c.t[t];
    if (!ti.src) return fail(KVRP_ERR_INVALID_ARG, "%s is NULL", names[t][0]);
    if (!aligned16(ti.src)) return fail(KVRP_ERR_ALIGNMENT, "%s is not 16-byte aligned", names[t][0]);
    if (c.rank > 0) {
      if (!ti.u || !ti.w) return fail(KVRP_ERR_INVALID_ARG, "rank > 0 needs both patch factors");
      if (!aligned16(ti.u) || !aligned16(ti.w))
        return fail(KVRP_ERR_ALIGNMENT, "patch factors must be 16-byte aligned");
    } else if (ti.u || ti.w) {
      return fail(KVRP_ERR_INVALID_ARG, "patch factors given with rank 0");
    }
    kvrp_status st = check_dst(&ti.dst, t == 0 ? "k_dst" : "v_dst", c.n_tokens, sh);
    if (st != KVRP_OK) return st;
  }
  return KVRP_OK;
}

// ---------------------------------------------------------------------------
// Plan builder
// ---------------------------------------------------------------------------
struct MapKey {
  const void* base;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3];
  int swz;
  bool operator<(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) < 0; }
};

// Process-wide caches of encoded tensor maps and phase tables.  A serving
// loop relocates into the same pools from the same canonical stores again and
// again; encoding a map costs about a microsecond, and a batch needs hundreds.
// The key holds every encoding parameter, so a hit is always the descriptor
// the driver would produce.  Both caches are bounded and simply start over
// when full.
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof(MapKey); ++i) h = (h ^ p[i]) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};
struct MapKeyEq {
  bool operator()(const MapKey& a, const MapKey& b) const { return std::memcmp(&a, &b, sizeof(MapKey)) == 0; }
};
struct TableKey {             // zero-filled before use, so it compares and hashes as bytes
  int64_t delta[3];
  int32_t sections[3];
  int32_t rot_dim;
  double theta;
  bool operator==(const TableKey& o) const { return std::memcmp(this, &o, sizeof(TableKey)) == 0; }
  bool operator<(const TableKey& o) const { return std::memcmp(this, &o, sizeof(TableKey)) < 0; }
};
struct TableKeyHash {
  size_t operator()(const TableKey& k) const {
    const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof(TableKey); ++i) h = (h ^ p[i]) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};
TableKey table_key(const int64_t delta[3], const int32_t sections[3], int rot_dim, double theta) {
  TableKey k;
  std::memset(&k, 0, sizeof(k));
  for (int i = 0; i < 3; ++i) {
    k.delta[i] = delta[i];
    k.sections[i] = sections[i];
  }
  k.rot_dim = rot_dim;
  k.theta = theta;
  return k;
}
struct CachedTable {
  float4 v[kTablePairs];
};
constexpr size_t kCacheMaxEntries = 16384;
std::mutex g_cache_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash, MapKeyEq> g_map_cache;
std::unordered_map<TableKey, CachedTable, TableKeyHash> g_table_cache;

class PlanBuilder {
 public:
  explicit PlanBuilder(const Shape& sh) : sh_(sh) {}

  kvrp_status map(const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_elems,
                  uint64_t s2_elems, uint32_t b0, uint32_t b1, CUtensorMapSwizzle swz, int32_t* idx) {
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.base = base;
    k.dims[0] = d0; k.dims[1] = d1; k.dims[2] = d2;
    k.strides[0] = s1_elems * 2; k.strides[1] = s2_elems * 2;
    k.box[0] = b0; k.box[1] = b1; k.box[2] = 1;
    k.swz = static_cast<int>(swz);
    auto found = map_index_.find(k);
    if (found != map_index_.end()) {
      *idx = found->second;
      return KVRP_OK;
    }
    CUtensorMap m;
    bool cached = false;
    {
      std::lock_guard<std::mutex> lk(g_cache_mu);
      auto hit = g_map_cache.find(k);
      if (hit != g_map_cache.end()) {
        m = hit->second;
        cached = true;
      }
    }
    if (!cached) {
      const cuuint32_t estr[3] = {1, 1, 1};
      const CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), k.dims,
                                  k.strides, k.box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS)
        return fail(KVRP_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d) for dims %llu x %llu x %llu",
                    (int)r, (unsigned long long)d0, (unsigned long long)d1, (unsigned long long)d2);
      std::lock_guard<std::mutex> lk(g_cache_mu);
      if (g_map_cache.size() >= kCacheMaxEntries) g_map_cache.clear();
      g_map_cache.emplace(k, m);
    }
    *idx = static_cast<int32_t>(maps_.size());
    maps_.push_back(m);
    map_index_[k] = *idx;
    return KVRP_OK;
  }

  int32_t table(const int64_t delta[3], const int32_t sections[3]) {
    const TableKey key = table_key(delta, sections, sh_.rot_dim, sh_.theta);
    auto f = tab_index_.find(key);
    if (f != tab_index_.end()) return f->second;
    const int32_t idx = static_cast<int32_t>(tabs_.size() / kTablePairs);
    tabs_.resize(tabs_.size() + kTablePairs);
    bool cached = false;
    {
      std::lock_guard<std::mutex> lk(g_cache_mu);
      auto hit = g_table_cache.find(key);
      if (hit != g_table_cache.end()) {
        std::memcpy(&tabs_[idx * kTablePairs], hit->second.v, sizeof(CachedTable));
        cached = true;
      }
    }
    if (!cached) {
      phase_table(delta, sections, sh_.theta, sh_.rot_dim, &tabs_[idx * kTablePairs]);
      CachedTable t;
      std::memcpy(t.v, &tabs_[idx * kTablePairs], sizeof(CachedTable));
      std::lock_guard<std::mutex> lk(g_cache_mu);
      if (g_table_cache.size() >= kCacheMaxEntries) g_table_cache.clear();
      g_table_cache.emplace(key, t);
    }
    tab_index_[key] = idx;
    return idx;
  }

  kvrp_status add(const ChunkIn& c) {
    ChunkRec r;
    std::memset(&r, 0, sizeof(r));
    r.n_tokens = c.n_tokens;
    r.rank = c.rank;
    r.n_tensors = c.n_tensors;
    r.table = -1;
    bool any_rot = false;
    const uint64_t L = static_cast<uint64_t>(sh_.n_layers);
    const uint64_t T = static_cast<uint64_t>(std::max(c.n_tokens, 1));
    for (int t = 0; t < c.n_tensors; ++t) {
      const TensorIn& ti = c.t[t];
      TensorRec& tr = r.t[t];
      tr.map_x = tr.map_u = tr.map_w = tr.map_dst = -1;
      tr.block_table = ti.dst.block_table;
      tr.dst = static_cast<uint16_t*>(ti.dst.base);
      tr.dst_layer_stride = ti.dst.layer_stride;
      tr.dst_start = ti.dst.dst_start;
      tr.num_pages = ti.dst.num_pages;
      tr.rot_kind = ti.rot_kind;
      tr.rot_from = ti.rot_from;
      any_rot |= ti.rot_kind != kRotNone;
      const int lead = static_cast<int>(ti.dst.dst_start % kPage);
      tr.n_tblk = c.n_tokens > 0 ? (lead + c.n_tokens + kTileRows - 1) / kTileRows : 0;
      if (c.n_tokens == 0) continue;
      const uint64_t sls = c.src_layer_stride ? c.src_layer_stride : T * sh_.D;
      // join the previous chunk's source group when these rows continue it
      XGroup* g = groups_[t].empty() ? nullptr : &groups_[t].back();
      const unsigned char* src = static_cast<const unsigned char*>(ti.src);
      // (the group's rows of one layer must stay within one layer stride, so
      // that every row the map spans belongs to one of its chunks)
      if (g && src == g->base + g->rows * sh_.D * 2 && g->rows + T <= (1ull << 30) &&
          (sh_.n_layers == 1 || (g->sls == sls && (g->rows + T) * sh_.D <= sls))) {
        tr.x_row0 = static_cast<int32_t>(g->rows);
        g->rows += T;
      } else {
        groups_[t].push_back(XGroup{src, sls, T});
        tr.x_row0 = 0;
      }
      tr.map_x = static_cast<int32_t>(groups_[t].size() - 1);   // a group index until finish()
      kvrp_status st;
      const uint64_t rows = static_cast<uint64_t>(ti.dst.num_pages) * kPage;
      const uint64_t dls = ti.dst.layer_stride ? ti.dst.layer_stride : rows * sh_.D;
      st = map(ti.dst.base, sh_.D, rows, L, sh_.D, dls, kBoxCols, kPage, CU_TENSOR_MAP_SWIZZLE_128B,
               &tr.map_dst);
      if (st != KVRP_OK) return st;
      if (c.rank > 0) {
        const uint64_t m = static_cast<uint64_t>(c.rank);
        const uint64_t uls = c.u_layer_stride ? c.u_layer_stride : T * m;
        const uint64_t wls = c.w_layer_stride ? c.w_layer_stride : (uint64_t)sh_.D * m;
        st = map(ti.u, m, T, L, m, uls, 16, kTileRows, CU_TENSOR_MAP_SWIZZLE_32B, &tr.map_u);
        if (st != KVRP_OK) return st;
        st = map(ti.w, m, sh_.D, L, m, wls, 16, kBoxCols, CU_TENSOR_MAP_SWIZZLE_32B, &tr.map_w);
        if (st != KVRP_OK) return st;
      }
    }
    if (any_rot && c.n_tokens > 0) r.table = table(c.delta, c.sections);
    // shared memory and TMA boxes work in steps of 16 ranks; the boxes of a
    // rank-8 tail reach past the factor's last column and read zeros there
    m_max_ = std::max(m_max_, (c.rank + 15) / 16 * 16);
    chunks_.push_back(r);
    return KVRP_OK;
  }

  // Chooses the item granularity and pipeline depth and serialises the plan.
  kvrp_status finish(int sms, int smem_optin, uint32_t* status, std::vector<unsigned char>* out,
                     int* grid, int* smem_bytes) {
    // one source map per group of consecutive chunks (see TensorRec::x_row0)
    for (int t = 0; t < 2; ++t) {
      std::vector<int32_t> gmap(groups_[t].size());
      for (size_t i = 0; i < groups_[t].size(); ++i) {
        const XGroup& g = groups_[t][i];
        // one layer: the stride is never followed; keep it at least one layer of the group's rows
        const uint64_t sls = sh_.n_layers == 1 ? std::max<uint64_t>(g.sls, g.rows * sh_.D) : g.sls;
        const kvrp_status st = map(g.base, sh_.D, g.rows, static_cast<uint64_t>(sh_.n_layers), sh_.D, sls,
                                   kBoxCols, kTileRows, CU_TENSOR_MAP_SWIZZLE_128B, &gmap[i]);
        if (st != KVRP_OK) return st;
      }
      for (ChunkRec& r : chunks_)
        if (t < r.n_tensors && r.n_tokens > 0) r.t[t].map_x = gmap[r.t[t].map_x];
    }
    PlanHdr h;
    std::memset(&h, 0, sizeof(h));
    h.n_chunks = static_cast<int32_t>(chunks_.size());
    h.D = sh_.D;
    h.n_layers = sh_.n_layers;
    h.n_sub = (sh_.D + kSubCols - 1) / kSubCols;
    h.m_max = m_max_;
    h.status = status;
    h.wait_cycles = test_wait_limit();
    // item granularity: whole rows unless that leaves SMs idle
    int64_t tiles = 0;
    for (const ChunkRec& r : chunks_)
      for (int t = 0; t < r.n_tensors; ++t) tiles += (int64_t)r.t[t].n_tblk * sh_.n_layers;
    int spi = h.n_sub;
    while (spi > 1 && tiles * ((h.n_sub + spi - 1) / spi) < 2ll * sms) spi = (spi + 1) / 2;
    h.subs_per_item = spi;
    h.n_sg = (h.n_sub + spi - 1) / spi;
    // tile prefix sums per tensor; items enumerate (tensor, layer, tile, group)
    h.n_tensors = chunks_.empty() ? 0 : chunks_[0].n_tensors;
    std::vector<int32_t> tbeg;
    int64_t items = 0;
    for (int t = 0; t < h.n_tensors; ++t) {
      int64_t tiles_t = 0;
      for (const ChunkRec& r : chunks_) {
        tbeg.push_back(static_cast<int32_t>(tiles_t));
        tiles_t += r.t[t].n_tblk;
      }
      tbeg.push_back(static_cast<int32_t>(tiles_t));
      if (tiles_t > (1ll << 30)) return fail(KVRP_ERR_INVALID_ARG, "too many tiles in one launch");
      h.tiles[t] = static_cast<int32_t>(tiles_t);
      const int64_t n = tiles_t * sh_.n_layers * h.n_sg;
      if (t == 0) h.items0 = static_cast<int32_t>(std::min<int64_t>(n, INT32_MAX));
      items += n;
    }
    if (items > (1ll << 31) - 1) return fail(KVRP_ERR_INVALID_ARG, "too many tiles in one launch");
    h.n_items = static_cast<int32_t>(items);
    // pipeline depth from the shared-memory budget (and TMEM: 128 columns a stage)
    const int budget = smem_optin - 1024;
    const int n_tables = static_cast<int>(tabs_.size() / kTablePairs);
    // Preference order: deeper pipeline, double-buffered U, then tables in
    // shared memory (one fixed copy, or one per stage), else global tables.
    int stages = 0, u_bufs = 0, tab_mode = kTabGlobal;
    const int modes_multi[2] = {kTabStaged, kTabGlobal};
    const int modes_single[1] = {kTabFixed};
    const int* modes = n_tables <= 1 ? modes_single : modes_multi;
    const int n_modes = n_tables <= 1 ? 1 : 2;
    for (int s = kMaxStages - kMaxStages % kEpiGroups; s >= kEpiGroups && stages == 0; s -= kEpiGroups) {
      for (int ub = 2; ub >= 1 && stages == 0; --ub) {
        for (int mi = 0; mi < n_modes && stages == 0; ++mi) {
          if ((int)smem_layout(m_max_, s, ub, modes[mi]).total <= budget) {
            stages = s;
            u_bufs = ub;
            tab_mode = modes[mi];
          }
        }
      }
    }
    if (stages == 0) return fail(KVRP_ERR_UNSUPPORTED, "rank %d does not fit in shared memory", m_max_);
    h.stages = stages;
    h.u_bufs = u_bufs;
    h.n_tables = n_tables;
    h.tab_mode = tab_mode;
    h.tmem_cols = 0;
    if (m_max_ > 0) {
      h.tmem_cols = 32;
      while (h.tmem_cols < kAccSlots * kSubCols) h.tmem_cols *= 2;
    }
    auto align = [](size_t v) { return (v + 127) & ~static_cast<size_t>(127); };
    size_t off = align(sizeof(PlanHdr));
    h.off_maps = static_cast<uint32_t>(off);
    off = align(off + maps_.size() * sizeof(CUtensorMap));
    h.off_tabs = static_cast<uint32_t>(off);
    off = align(off + tabs_.size() * sizeof(float4));
    h.off_chunks = static_cast<uint32_t>(off);
    off = align(off + chunks_.size() * sizeof(ChunkRec));
    h.off_tbeg = static_cast<uint32_t>(off);
    off = align(off + tbeg.size() * sizeof(int32_t));
    h.total_bytes = static_cast<uint32_t>(off);
    out->assign(off, 0);
    std::memcpy(out->data(), &h, sizeof(h));
    if (!maps_.empty()) std::memcpy(out->data() + h.off_maps, maps_.data(), maps_.size() * sizeof(CUtensorMap));
    if (!tabs_.empty()) std::memcpy(out->data() + h.off_tabs, tabs_.data(), tabs_.size() * sizeof(float4));
    std::memcpy(out->data() + h.off_chunks, chunks_.data(), chunks_.size() * sizeof(ChunkRec));
    if (!tbeg.empty()) std::memcpy(out->data() + h.off_tbeg, tbeg.data(), tbeg.size() * sizeof(int32_t));
    *grid = static_cast<int>(std::min<int64_t>(items, sms));
    *smem_bytes = static_cast<int>(smem_layout(m_max_, stages, u_bufs, tab_mode).total) + 1024;
    return KVRP_OK;
  }

 private:
  Shape sh_;
  int m_max_ = 0;
  std::vector<CUtensorMap> maps_;
  std::map<MapKey, int32_t> map_index_;
  std::vector<float4> tabs_;
  std::map<TableKey, int32_t> tab_index_;
  std::vector<ChunkRec> chunks_;
  struct XGroup {
    const unsigned char* base;   // first row of the group's first chunk (layer 0)
    uint64_t sls;                // layer stride, elements
    uint64_t rows;               // rows of all the group's chunks
  };
  std::vector<XGroup> groups_[2];   // per tensor, in chunk order
};

// Builds the plan for `chunks` and launches it: as a kernel parameter when it
// fits, otherwise through `workspace` (device), carried there by upload_plan.
kvrp_status run(const Shape& sh, const std::vector<ChunkIn>& chunks, uint32_t* d_status, void* workspace,
                size_t workspace_bytes, cudaStream_t stream);

}  // namespace

uint32_t test_wait_limit() { return g_test_wait_limit.load(std::memory_order_relaxed); }

kvrp_status current_device_sms(int* sms, int* smem_optin) {
  DeviceInfo* di = nullptr;
  const kvrp_status st = device_info(&di);
  if (st != KVRP_OK) return st;
  *sms = di->sms;
  *smem_optin = di->smem_optin;
  return KVRP_OK;
}

namespace {

kvrp_status run(const Shape& sh, const std::vector<ChunkIn>& chunks, uint32_t* d_status, void* workspace,
                size_t workspace_bytes, cudaStream_t stream) {
  DeviceInfo* di = nullptr;
  kvrp_status st = device_info(&di);
  if (st != KVRP_OK) return st;
  PlanBuilder pb(sh);
  for (const ChunkIn& c : chunks) {
    st = pb.add(c);
    if (st != KVRP_OK) return st;
  }
  std::vector<unsigned char> bytes;
  int grid = 0, smem = 0;
  g_last_launches = 0;
  st = pb.finish(di->sms, di->smem_optin, d_status, &bytes, &grid, &smem);
  if (st != KVRP_OK) return st;
  if (grid == 0) return KVRP_OK;  // nothing to move
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (di->prepared_smem < smem) {
      const cudaError_t e = prepare_kernel(di->smem_optin);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
      di->prepared_smem = di->smem_optin;
    }
  }
  cudaError_t e;
  if (workspace == nullptr) {
    if (bytes.size() > (size_t)kParamPlanBytes)
      return fail(KVRP_ERR_INVALID_ARG, "internal: single-chunk plan exceeds the parameter block");
    std::vector<unsigned char> padded(kParamPlanBytes, 0);
    std::memcpy(padded.data(), bytes.data(), bytes.size());
    e = launch_relocate(padded.data(), nullptr, grid, smem, stream);
  } else {
    if (bytes.size() > workspace_bytes)
      return fail(KVRP_ERR_WORKSPACE, "workspace holds %zu bytes, the plan needs %zu", workspace_bytes,
                  bytes.size());
    e = upload_plan(bytes.data(), bytes.size(), workspace, stream);
    if (e != cudaSuccess) return cuda_fail(e, "plan upload");
    g_last_launches = upload_launches(bytes.size());
    e = launch_relocate(nullptr, workspace, grid, smem, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  g_last_launches += 1;
  return KVRP_OK;
}

void set_plain_shift(ChunkIn* c, int64_t delta, int rot_dim) {
  c->delta[0] = delta;
  c->delta[1] = c->delta[2] = 0;
  c->sections[0] = rot_dim / 2;
  c->sections[1] = c->sections[2] = 0;
}

TensorIn tensor_in(const void* src, const void* u, const void* w, const kvrp_dst* d, int rot_kind,
                   int rot_from) {
  TensorIn t;
  t.src = src;
  t.u = u;
  t.w = w;
  t.dst = d ? *d : kvrp_dst{};
  t.rot_kind = rot_kind;
  t.rot_from = rot_from;
  return t;
}

// The allocation-free batch path: same plan and kernel as kv_relocate_batch,
// but the plan goes to the library's fixed device array, carried there by the
// same parameter-block copy kernels; nothing is allocated on the device or
// pinned on the host.
kvrp_status run_noalloc(const Shape& sh, const std::vector<ChunkIn>& chunks, uint32_t* d_status,
                        cudaStream_t stream) {
  DeviceInfo* di = nullptr;
  kvrp_status st = device_info(&di);
  if (st != KVRP_OK) return st;
  PlanBuilder pb(sh);
  for (const ChunkIn& c : chunks) {
    st = pb.add(c);
    if (st != KVRP_OK) return st;
  }
  std::vector<unsigned char> bytes;
  int grid = 0, smem = 0;
  g_last_launches = 0;
  st = pb.finish(di->sms, di->smem_optin, d_status, &bytes, &grid, &smem);
  if (st != KVRP_OK) return st;
  if (grid == 0) return KVRP_OK;
  if (bytes.size() > noalloc_scratch_bytes())
    return fail(KVRP_ERR_WORKSPACE, "plan of %zu bytes exceeds the fixed %zu-byte device array", bytes.size(),
                noalloc_scratch_bytes());
  void* scratch = nullptr;
  cudaError_t e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(fixed plan array)");
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (di->prepared_smem < smem) {
      e = prepare_kernel(di->smem_optin);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
      di->prepared_smem = di->smem_optin;
    }
  }
  e = upload_plan(bytes.data(), bytes.size(), scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "plan upload to the fixed array");
  g_last_launches = upload_launches(bytes.size());
  e = launch_relocate(nullptr, scratch, grid, smem, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  g_last_launches += 1;
  return KVRP_OK;
}

// Prefixes the last error with the index of the chunk it came from.
kvrp_status chunk_error(int i, kvrp_status st) {
  std::string msg = "chunk " + std::to_string(i) + ": " + g_last_error;
  std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg.c_str());
  return st;
}

kvrp_status check_gqa_shape(int32_t n_layers, int32_t n_kv_heads, int32_t head_dim, double rope_theta) {
  if (n_layers <= 0 || n_kv_heads <= 0) return fail(KVRP_ERR_INVALID_ARG, "n_layers and n_kv_heads must be > 0");
  if (head_dim != 64 && head_dim != 128) return fail(KVRP_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (!(rope_theta > 0.0) || !std::isfinite(rope_theta)) return fail(KVRP_ERR_INVALID_ARG, "rope_theta must be > 0");
  if ((int64_t)n_kv_heads * head_dim > 65536) return fail(KVRP_ERR_UNSUPPORTED, "row too wide");
  return KVRP_OK;
}

kvrp_status check_mla_shape(int32_t n_layers, int32_t kv_lora_dim, int32_t rope_dim, double rope_theta) {
  if (n_layers <= 0) return fail(KVRP_ERR_INVALID_ARG, "n_layers must be > 0");
  if (rope_dim != 64) return fail(KVRP_ERR_UNSUPPORTED, "rope_dim must be 64");
  if (kv_lora_dim < 0 || kv_lora_dim % 64 != 0 || kv_lora_dim > 65536 - 64)
    return fail(KVRP_ERR_UNSUPPORTED, "kv_lora_dim must be a multiple of 64");
  if (!(rope_theta > 0.0) || !std::isfinite(rope_theta)) return fail(KVRP_ERR_INVALID_ARG, "rope_theta must be > 0");
  return KVRP_OK;
}

kvrp_status check_sections(const int32_t sec[3], int32_t head_dim) {
  if (!sec) return fail(KVRP_ERR_INVALID_ARG, "mrope_section is required");
  int64_t pairs = 0;
  for (int i = 0; i < 3; ++i) {
    if (sec[i] < 0) return fail(KVRP_ERR_INVALID_ARG, "mrope_section entries must be >= 0");
    pairs += sec[i];
  }
  if (pairs != head_dim / 2)
    return fail(KVRP_ERR_INVALID_ARG, "mrope_section must sum to head_dim / 2 = %d (got %lld)", head_dim / 2,
                (long long)pairs);
  return KVRP_OK;
}

// One GQA/MHA chunk of a batch: keys turn per head, values do not.
ChunkIn gqa_chunk(const kvrp_chunk& k, int32_t head_dim) {
  ChunkIn c;
  c.n_tensors = 2;
  c.t[0] = tensor_in(k.k_src, k.uk, k.vk, &k.k_dst, head_dim == 128 ? kRotHalf128 : kRotHalf64, 0);
  c.t[1] = tensor_in(k.v_src, k.uv, k.vv, &k.v_dst, kRotNone, 0);
  c.src_layer_stride = k.src_layer_stride;
  c.u_layer_stride = k.u_layer_stride;
  c.w_layer_stride = k.v_layer_stride;
  c.n_tokens = k.n_tokens;
  c.rank = k.rank;
  set_plain_shift(&c, k.delta, head_dim);
  return c;
}

// The checked chunk list of a GQA/MHA batch; under M-RoPE (delta_thw != NULL)
// chunk i turns by the shifts delta_thw[3i .. 3i + 2] of the sections `sec`.
kvrp_status gqa_batch(const kvrp_chunk* chunks, int32_t n_chunks, const Shape& sh, int32_t head_dim,
                      const int64_t* delta_thw, const int32_t* sec, std::vector<ChunkIn>* out) {
  out->resize(n_chunks);
  for (int i = 0; i < n_chunks; ++i) {
    ChunkIn& c = (*out)[i];
    c = gqa_chunk(chunks[i], head_dim);
    if (delta_thw) {
      for (int j = 0; j < 3; ++j) {
        c.delta[j] = delta_thw[3 * i + j];
        c.sections[j] = sec[j];
      }
    }
    const kvrp_status st = check_chunk(c, sh);
    if (st != KVRP_OK) return chunk_error(i, st);
  }
  return KVRP_OK;
}

kvrp_status check_workspace(void* workspace, size_t workspace_bytes, int32_t n_chunks) {
  if (!workspace) return fail(KVRP_ERR_WORKSPACE, "a batch call needs a device workspace");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(KVRP_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (workspace_bytes < plan_bytes_bound(n_chunks))
    return fail(KVRP_ERR_WORKSPACE, "workspace smaller than kv_relocate_batch_workspace_size(%d)", n_chunks);
  return KVRP_OK;
}

}  // namespace
}  // namespace kvrp

using namespace kvrp;

extern "C" {

kvrp_status kv_relocate_patch(const void* k_src, const void* v_src, int64_t src_layer_stride,
                              int32_t n_layers, int32_t n_tokens, int32_t n_kv_heads, int32_t head_dim,
                              int64_t delta, double rope_theta, int32_t rank, const void* uk,
                              const void* vk, const void* uv, const void* vv, int64_t u_layer_stride,
                              int64_t v_layer_stride, const kvrp_dst* k_dst, const kvrp_dst* v_dst,
                              uint32_t* d_status, kvrp_stream_t stream) {
  kvrp_status st = check_gqa_shape(n_layers, n_kv_heads, head_dim, rope_theta);
  if (st != KVRP_OK) return st;
  if (!k_dst || !v_dst) return fail(KVRP_ERR_INVALID_ARG, "k_dst and v_dst are required");
  const Shape sh{n_layers, n_kv_heads * head_dim, head_dim, rope_theta};
  ChunkIn c;
  c.n_tensors = 2;
  c.t[0] = tensor_in(k_src, uk, vk, k_dst, head_dim == 128 ? kRotHalf128 : kRotHalf64, 0);
  c.t[1] = tensor_in(v_src, uv, vv, v_dst, kRotNone, 0);
  c.src_layer_stride = src_layer_stride;
  c.u_layer_stride = u_layer_stride;
  c.w_layer_stride = v_layer_stride;
  c.n_tokens = n_tokens;
  c.rank = rank;
  set_plain_shift(&c, delta, head_dim);
  st = check_chunk(c, sh);
  if (st != KVRP_OK) return st;
  return run(sh, {c}, d_status, nullptr, 0, stream);
}

kvrp_status kv_relocate_patch_mrope(const void* k_src, const void* v_src, int64_t src_layer_stride,
                                    int32_t n_layers, int32_t n_tokens, int32_t n_kv_heads, int32_t head_dim,
                                    const int64_t delta_thw[3], const int32_t mrope_section[3],
                                    double rope_theta, int32_t rank, const void* uk, const void* vk,
                                    const void* uv, const void* vv, int64_t u_layer_stride,
                                    int64_t v_layer_stride, const kvrp_dst* k_dst, const kvrp_dst* v_dst,
                                    uint32_t* d_status, kvrp_stream_t stream) {
  kvrp_status st = check_gqa_shape(n_layers, n_kv_heads, head_dim, rope_theta);
  if (st != KVRP_OK) return st;
  if (!k_dst || !v_dst) return fail(KVRP_ERR_INVALID_ARG, "k_dst and v_dst are required");
  if (!delta_thw) return fail(KVRP_ERR_INVALID_ARG, "delta_thw is required");
  st = check_sections(mrope_section, head_dim);
  if (st != KVRP_OK) return st;
  const Shape sh{n_layers, n_kv_heads * head_dim, head_dim, rope_theta};
  ChunkIn c;
  c.n_tensors = 2;
  c.t[0] = tensor_in(k_src, uk, vk, k_dst, head_dim == 128 ? kRotHalf128 : kRotHalf64, 0);
  c.t[1] = tensor_in(v_src, uv, vv, v_dst, kRotNone, 0);
  c.src_layer_stride = src_layer_stride;
  c.u_layer_stride = u_layer_stride;
  c.w_layer_stride = v_layer_stride;
  c.n_tokens = n_tokens;
  c.rank = rank;
  for (int i = 0; i < 3; ++i) {
    c.delta[i] = delta_thw[i];
    c.sections[i] = mrope_section[i];
  }
  st = check_chunk(c, sh);
  if (st != KVRP_OK) return st;
  return run(sh, {c}, d_status, nullptr, 0, stream);
}

kvrp_status kv_relocate_patch_mla(const void* src, int64_t src_layer_stride, int32_t n_layers,
                                  int32_t n_tokens, int32_t kv_lora_dim, int32_t rope_dim, int64_t delta,
                                  double rope_theta, int32_t rank, const void* u, const void* v,
                                  int64_t u_layer_stride, int64_t v_layer_stride, const kvrp_dst* dst,
                                  uint32_t* d_status, kvrp_stream_t stream) {
  kvrp_status st = check_mla_shape(n_layers, kv_lora_dim, rope_dim, rope_theta);
  if (st != KVRP_OK) return st;
  if (!dst) return fail(KVRP_ERR_INVALID_ARG, "dst is required");
  const Shape sh{n_layers, kv_lora_dim + rope_dim, rope_dim, rope_theta};
  ChunkIn c;
  c.n_tensors = 1;
  c.t[0] = tensor_in(src, u, v, dst, kRotHalf64, kv_lora_dim);
  c.t[1] = tensor_in(nullptr, nullptr, nullptr, nullptr, kRotNone, 0);
  c.src_layer_stride = src_layer_stride;
  c.u_layer_stride = u_layer_stride;
  c.w_layer_stride = v_layer_stride;
  c.n_tokens = n_tokens;
  c.rank = rank;
  set_plain_shift(&c, delta, rope_dim);
  st = check_chunk(c, sh);
  if (st != KVRP_OK) return st;
  return run(sh, {c}, d_status, nullptr, 0, stream);
}

size_t kv_relocate_batch_workspace_size(int32_t n_chunks) {
  if (n_chunks <= 0) return 0;
  return plan_bytes_bound(n_chunks);
}

kvrp_status kv_relocate_batch(const kvrp_chunk* chunks, int32_t n_chunks, int32_t n_layers, int32_t n_kv_heads,
                              int32_t head_dim, double rope_theta, void* workspace, size_t workspace_bytes,
                              uint32_t* d_status, kvrp_stream_t stream) {
  if (n_chunks < 0 || (n_chunks > 0 && !chunks)) return fail(KVRP_ERR_INVALID_ARG, "bad chunk array");
  if (n_chunks == 0) return KVRP_OK;
  kvrp_status st = check_gqa_shape(n_layers, n_kv_heads, head_dim, rope_theta);
  if (st != KVRP_OK) return st;
  st = check_workspace(workspace, workspace_bytes, n_chunks);
  if (st != KVRP_OK) return st;
  const Shape sh{n_layers, n_kv_heads * head_dim, head_dim, rope_theta};
  std::vector<ChunkIn> in;
  st = gqa_batch(chunks, n_chunks, sh, head_dim, nullptr, nullptr, &in);
  if (st != KVRP_OK) return st;
  return run(sh, in, d_status, workspace, workspace_bytes, stream);
}

kvrp_status kv_relocate_batch_mrope(const kvrp_chunk* chunks, const int64_t* delta_thw, int32_t n_chunks,
                                    int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
                                    const int32_t mrope_section[3], double rope_theta, void* workspace,
                                    size_t workspace_bytes, uint32_t* d_status, kvrp_stream_t stream) {
  if (n_chunks < 0 || (n_chunks > 0 && (!chunks || !delta_thw))) return fail(KVRP_ERR_INVALID_ARG, "bad chunk array");
  if (n_chunks == 0) return KVRP_OK;
  kvrp_status st = check_gqa_shape(n_layers, n_kv_heads, head_dim, rope_theta);
  if (st != KVRP_OK) return st;
  st = check_sections(mrope_section, head_dim);
  if (st != KVRP_OK) return st;
  st = check_workspace(workspace, workspace_bytes, n_chunks);
  if (st != KVRP_OK) return st;
  const Shape sh{n_layers, n_kv_heads * head_dim, head_dim, rope_theta};
  std::vector<ChunkIn> in;
  st = gqa_batch(chunks, n_chunks, sh, head_dim, delta_thw, mrope_section, &in);
  if (st != KVRP_OK) return st;
  return run(sh, in, d_status, workspace, workspace_bytes, stream);
}

kvrp_status kv_relocate_batch_mla(const kvrp_mla_chunk* chunks, int32_t n_chunks, int32_t n_layers,
                                  int32_t kv_lora_dim, int32_t rope_dim, double rope_theta, void* workspace,
                                  size_t workspace_bytes, uint32_t* d_status, kvrp_stream_t stream) {
  if (n_chunks < 0 || (n_chunks > 0 && !chunks)) return fail(KVRP_ERR_INVALID_ARG, "bad chunk array");
  if (n_chunks == 0) return KVRP_OK;
  kvrp_status st = check_mla_shape(n_layers, kv_lora_dim, rope_dim, rope_theta);
  if (st != KVRP_OK) return st;
  st = check_workspace(workspace, workspace_bytes, n_chunks);
  if (st != KVRP_OK) return st;
  const Shape sh{n_layers, kv_lora_dim + rope_dim, rope_dim, rope_theta};
  std::vector<ChunkIn> in(n_chunks);
  for (int i = 0; i < n_chunks; ++i) {
    const kvrp_mla_chunk& k = chunks[i];
    ChunkIn& c = in[i];
    c.n_tensors = 1;
    c.t[0] = tensor_in(k.src, k.u, k.v, &k.dst, kRotHalf64, kv_lora_dim);
    c.t[1] = tensor_in(nullptr, nullptr, nullptr, nullptr, kRotNone, 0);
    c.src_layer_stride = k.src_layer_stride;
    c.u_layer_stride = k.u_layer_stride;
    c.w_layer_stride = k.v_layer_stride;
    c.n_tokens = k.n_tokens;
    c.rank = k.rank;
    set_plain_shift(&c, k.delta, rope_dim);
    st = check_chunk(c, sh);
    if (st != KVRP_OK) return chunk_error(i, st);
  }
  return run(sh, in, d_status, workspace, workspace_bytes, stream);
}

kvrp_status kv_relocate_batch_noalloc(const kvrp_chunk* chunks, int32_t n_chunks, int32_t n_layers,
                                      int32_t n_kv_heads, int32_t head_dim, double rope_theta,
                                      uint32_t* d_status, kvrp_stream_t stream) {
  if (n_chunks < 0 || (n_chunks > 0 && !chunks)) return fail(KVRP_ERR_INVALID_ARG, "bad chunk array");
  if (n_chunks > KVRP_NOALLOC_MAX_CHUNKS)
    return fail(KVRP_ERR_INVALID_ARG, "kv_relocate_batch_noalloc takes at most %d chunks (got %d)",
                KVRP_NOALLOC_MAX_CHUNKS, n_chunks);
  if (n_chunks == 0) return KVRP_OK;
  kvrp_status st = check_gqa_shape(n_layers, n_kv_heads, head_dim, rope_theta);
  if (st != KVRP_OK) return st;
  const Shape sh{n_layers, n_kv_heads * head_dim, head_dim, rope_theta};
  std::vector<ChunkIn> in;
  st = gqa_batch(chunks, n_chunks, sh, head_dim, nullptr, nullptr, &in);
  if (st != KVRP_OK) return st;
  return run_noalloc(sh, in, d_status, stream);
}

void kvrp_test_set_wait_limit(uint32_t cycles) { g_test_wait_limit.store(cycles, std::memory_order_relaxed); }

const char* kvrp_status_string(kvrp_status status) {
  switch (status) {
    case KVRP_OK: return "KVRP_OK";
    case KVRP_ERR_INVALID_ARG: return "KVRP_ERR_INVALID_ARG";
    case KVRP_ERR_ALIGNMENT: return "KVRP_ERR_ALIGNMENT";
    case KVRP_ERR_UNSUPPORTED: return "KVRP_ERR_UNSUPPORTED";
    case KVRP_ERR_CUDA: return "KVRP_ERR_CUDA";
    case KVRP_ERR_WORKSPACE: return "KVRP_ERR_WORKSPACE";
  }
  return "KVRP_ERR_UNKNOWN";
}

const char* kvrp_last_error(void) { return g_last_error; }

int32_t kvrp_last_launch_count(void) { return g_last_launches; }

int32_t kvrp_version(void) { return 100; }

}  // extern "C"
