/*
 * kvrp.h -- C ABI of the GB300 KV relocation + rank-m patch library (libkvrp.so).
 *
 * The operator (Kamera, gist.science/pt/paper/2606.23581, section 2 "O Operador
 * Kamera"; the Korean summary gist.science/ko/paper/2606.23581 section 2 states
 * the same) reuses a chunk B that was cached on its own, KV(B|empty), at a new
 * position after a new antecedent A:
 *
 *     KV^(B|A) = R(delta) . KV(B|empty) + U_m V_m^T
 *
 *   R(delta)   exact RoPE re-rotation of the cached keys by the position shift
 *              delta (new position - old position), rotate-half convention:
 *              feature i of a rotated head pairs with feature i + d/2 and the
 *              pair turns by delta * theta^(-2i/d).  Values are not rotated
 *              (GQA/MHA); for MLA only the 64-dim k_rope is turned and c_KV is
 *              reused byte for byte (section 2, family bullets).
 *   U_m V_m^T  rank-m conditioning patch, added after the rotation, to K and
 *              to V (each tensor has its own factor pair), or to the whole
 *              576-wide MLA row (one pair).
 *
 * The result is rounded to bf16 and written straight into a paged KV cache:
 * token t of a chunk lands at position q = dst_start + t of its sequence,
 * physical page block_table[q / 16], slot q % 16.
 *
 * Conventions shared by every entry point
 *   - bf16 data is passed as raw pointers (uint16 bit patterns).  Rows are
 *     dense: a token row of one tensor is D contiguous bf16 values, with
 *     D = n_kv_heads * head_dim (GQA/MHA) or kv_lora_dim + rope_dim (MLA).
 *   - Canonical source of one tensor: [n_layers][n_tokens][D]; layer l starts
 *     at src + l * src_layer_stride (elements).
 *   - Patch factors of one tensor: U_m [n_layers][n_tokens][rank] (token-major)
 *     and V_m [n_layers][D][rank] (feature-major); layer strides in elements.
 *     Singular values are expected to be folded into U_m.
 *   - Destination pool of one tensor: layer l at base + l * layer_stride,
 *     laid out [num_pages][16][D].  A NULL block_table means a contiguous
 *     destination (identity table: position q is row q of the layer).
 *   - Every device pointer is owned by the caller, must be 16-byte aligned
 *     (block tables: 4-byte aligned) and must stay valid until the stream work
 *     is done.  Strides and dst_start are in elements; strides must be
 *     multiples of 8 elements.
 *   - rank must be 0 or a multiple of 8 up to 128 (the factor rows are then a
 *     multiple of 16 bytes, as the TMA copies need); head_dim must be 64 or
 *     128; MLA rope_dim must be 64 and kv_lora_dim a multiple of 64.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Host-detected problems are returned as kvrp_status before anything is
 *     enqueued.  Problems only the device can see are OR-ed into *d_status
 *     (optional, device memory, read it after synchronising):
 *     KVRP_DEV_BAD_PAGE: a block-table entry was outside [0, num_pages); the
 *     rows of that page were skipped.  KVRP_DEV_TIMEOUT: an internal pipeline
 *     wait gave up (it is bounded); the output is incomplete.
 *   - Destination slots written by one call must not overlap (a bijective
 *     block table); overlapping slots give an unspecified winner.  Source and
 *     destination must not overlap.
 *   - Thread safety: calls may come from several host threads.
 */
#ifndef KVRP_H
#define KVRP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* kvrp_stream_t;

typedef enum kvrp_status {
  KVRP_OK = 0,
  KVRP_ERR_INVALID_ARG = 1,   /* a NULL pointer, a size or stride out of range      */
  KVRP_ERR_ALIGNMENT = 2,     /* a pointer or stride breaks the 16-byte rule        */
  KVRP_ERR_UNSUPPORTED = 3,   /* head_dim / rank / rope_dim outside the kernel's set */
  KVRP_ERR_CUDA = 4,          /* a CUDA runtime or driver call failed               */
  KVRP_ERR_WORKSPACE = 5      /* the batch workspace is missing or too small        */
} kvrp_status;

#define KVRP_DEV_BAD_PAGE 0x1u
#define KVRP_DEV_TIMEOUT 0x2u

/* One destination pool (one tensor). */
typedef struct kvrp_dst {
  void* base;                 /* bf16 pool; layer l at base + l * layer_stride          */
  int64_t layer_stride;       /* elements between layers (>= num_pages * 16 * D)        */
  const int32_t* block_table; /* device int32, one entry per logical page of the
                                 sequence (>= ceil((dst_start + n_tokens) / 16)); NULL
                                 = contiguous                                            */
  int32_t num_pages;          /* physical pages per layer                               */
  int32_t page_size;          /* tokens per page; must be 16                            */
  int64_t dst_start;          /* sequence position of the chunk's first token (>= 0)    */
} kvrp_dst;

/*
 * kv_relocate_patch -- one GQA/MHA chunk, all layers, K and V, one launch.
 *   K gets R(delta) + U_K V_K^T; V gets V + U_V V_V^T (section 2, GQA bullet:
 *   relocate the full keys by re-applying RoPE, patch both K and V; the MHA
 *   bullet is the same with n_kv_heads = query heads).
 *   k_src, v_src  canonical K and V, [n_layers][n_tokens][D] at src_layer_stride.
 *   rank          m; 0 = relocation only (V is then copied byte for byte).
 *   uk, vk        U_m [L][T][m] and V_m [L][D][m] of the K patch (NULL iff rank 0).
 *   uv, vv        the same for the V patch.
 *   rope_theta    RoPE base (theta_i = rope_theta^(-2i/head_dim)).
 *   delta         position shift, new minus old.
 */
kvrp_status kv_relocate_patch(
    const void* k_src, const void* v_src, int64_t src_layer_stride,
    int32_t n_layers, int32_t n_tokens, int32_t n_kv_heads, int32_t head_dim,
    int64_t delta, double rope_theta, int32_t rank,
    const void* uk, const void* vk, const void* uv, const void* vv,
    int64_t u_layer_stride, int64_t v_layer_stride,
    const kvrp_dst* k_dst, const kvrp_dst* v_dst,
    uint32_t* d_status, kvrp_stream_t stream);

/*
 * kv_relocate_patch_mrope -- kv_relocate_patch under M-RoPE, the multimodal
 * RoPE of Qwen-VL-style models, which re-rotate image and video KV with it
 * (gist.science/pt/paper/2606.17107, section 4: transplanted image KV is
 * re-rotated with M-RoPE).  The head_dim / 2 frequency pairs form three
 * consecutive sections -- temporal, height, width -- of mrope_section[0..2]
 * pairs (Qwen2.5-VL with head_dim 128: {16, 24, 24}); pair i turns by
 * delta_thw[s] * theta^(-2i/head_dim), s being the section holding i.
 *   delta_thw      host array: the (temporal, height, width) position shift.
 *   mrope_section  host array: frequency pairs per section, summing to head_dim / 2.
 *   Everything else as kv_relocate_patch.  Equal shifts give plain RoPE.
 */
kvrp_status kv_relocate_patch_mrope(
    const void* k_src, const void* v_src, int64_t src_layer_stride,
    int32_t n_layers, int32_t n_tokens, int32_t n_kv_heads, int32_t head_dim,
    const int64_t delta_thw[3], const int32_t mrope_section[3],
    double rope_theta, int32_t rank,
    const void* uk, const void* vk, const void* uv, const void* vv,
    int64_t u_layer_stride, int64_t v_layer_stride,
    const kvrp_dst* k_dst, const kvrp_dst* v_dst,
    uint32_t* d_status, kvrp_stream_t stream);

/*
 * kv_relocate_patch_mla -- one MLA chunk, all layers, one launch (section 2,
 * MLA bullet: only the decoupled 64-dim k_rope is relocated, c_KV is reused
 * byte for byte, the patch goes to both channels).
 *   src   rows [n_layers][n_tokens][kv_lora_dim + rope_dim] = c_KV ++ k_rope.
 *   u, v  U_m [L][T][m] and V_m [L][kv_lora_dim + rope_dim][m] (NULL iff rank 0).
 *   With rank 0 the c_KV part of every row is copied bit for bit.
 */
kvrp_status kv_relocate_patch_mla(
    const void* src, int64_t src_layer_stride, int32_t n_layers, int32_t n_tokens,
    int32_t kv_lora_dim, int32_t rope_dim, int64_t delta, double rope_theta,
    int32_t rank, const void* u, const void* v,
    int64_t u_layer_stride, int64_t v_layer_stride,
    const kvrp_dst* dst, uint32_t* d_status, kvrp_stream_t stream);

/* One chunk of a batch: its own source, shift, patch and destination. */
typedef struct kvrp_chunk {
  const void* k_src;          /* [n_layers][n_tokens][D] at src_layer_stride            */
  const void* v_src;
  int64_t src_layer_stride;
  int32_t n_tokens;
  int32_t rank;               /* 0 = relocation only                                    */
  int64_t delta;
  const void* uk;             /* K patch U_m [L][T][m]; NULL iff rank 0                 */
  const void* vk;             /* K patch V_m [L][D][m]                                  */
  const void* uv;             /* V patch U_m                                            */
  const void* vv;             /* V patch V_m                                            */
  int64_t u_layer_stride;
  int64_t v_layer_stride;
  kvrp_dst k_dst;
  kvrp_dst v_dst;
} kvrp_chunk;

/*
 * kv_relocate_batch -- many GQA/MHA chunks, each with its own delta and patch,
 * in ONE relocation kernel launch (section 3, the three window operations:
 * reorder under an orbit patch, sliding-window survival with R(delta) alone,
 * recall of an evicted chunk with a fresh patch).
 *   chunks      host array of n_chunks descriptors (read before the call returns).
 *   workspace   device scratch of at least kv_relocate_batch_workspace_size(n_chunks)
 *               bytes, 256-byte aligned, owned by the caller.  The call writes the
 *               launch's descriptors there on `stream` (small copy kernels carry
 *               them in their parameters, ahead of the relocation kernel); do not
 *               reuse it for another purpose until the stream work is done.  Two
 *               batch calls may share one workspace only on the same stream.
 * The workspace size covers every batch call below (GQA/MHA, M-RoPE, MLA).
 */
size_t kv_relocate_batch_workspace_size(int32_t n_chunks);

kvrp_status kv_relocate_batch(
    const kvrp_chunk* chunks, int32_t n_chunks,
    int32_t n_layers, int32_t n_kv_heads, int32_t head_dim, double rope_theta,
    void* workspace, size_t workspace_bytes,
    uint32_t* d_status, kvrp_stream_t stream);

/*
 * kv_relocate_batch_mrope -- kv_relocate_batch under M-RoPE: a window of
 * image or video chunks of a Qwen-VL-style model, each moved by its own
 * (temporal, height, width) shift, in one launch (transplanted image KV is
 * re-rotated with M-RoPE: gist.science/pt/paper/2606.17107, section 4; the
 * window operations are those of Kamera, section 3).
 *   delta_thw      host array [n_chunks][3]: chunk i turns frequency pair p by
 *                  delta_thw[3i + s] * theta^(-2p/head_dim), s being the section
 *                  of p; the chunks' own .delta fields are not read.
 *   mrope_section  host array: frequency pairs per (t, h, w) section, summing to
 *                  head_dim / 2 (Qwen2.5-VL with head_dim 128: {16, 24, 24}).
 *   Everything else as kv_relocate_batch (same workspace size).
 */
kvrp_status kv_relocate_batch_mrope(
    const kvrp_chunk* chunks, const int64_t* delta_thw, int32_t n_chunks,
    int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
    const int32_t mrope_section[3], double rope_theta,
    void* workspace, size_t workspace_bytes,
    uint32_t* d_status, kvrp_stream_t stream);

/* One MLA chunk of a batch: its own source rows, shift, patch and destination. */
typedef struct kvrp_mla_chunk {
  const void* src;            /* rows [n_layers][n_tokens][kv_lora_dim + rope_dim] = c_KV ++ k_rope */
  int64_t src_layer_stride;
  int32_t n_tokens;
  int32_t rank;               /* 0 = relocation only (c_KV copied byte for byte)       */
  int64_t delta;
  const void* u;              /* U_m [L][T][m]; NULL iff rank 0                         */
  const void* v;              /* V_m [L][kv_lora_dim + rope_dim][m]                     */
  int64_t u_layer_stride;
  int64_t v_layer_stride;
  kvrp_dst dst;
} kvrp_mla_chunk;

/*
 * kv_relocate_batch_mla -- many MLA chunks, each with its own delta and patch,
 * in one launch: the window operations of Kamera section 3 (survival by
 * R(delta) alone, recall with a fresh patch) on a DeepSeek-style cache, where
 * only the k_rope tail of each row turns and c_KV is reused byte for byte
 * (section 2, MLA bullet: survival needs only R(delta) for GQA and MLA alike).
 *   Shapes and rules per chunk as kv_relocate_patch_mla; workspace as
 *   kv_relocate_batch (kv_relocate_batch_workspace_size(n_chunks) bytes).
 */
kvrp_status kv_relocate_batch_mla(
    const kvrp_mla_chunk* chunks, int32_t n_chunks, int32_t n_layers,
    int32_t kv_lora_dim, int32_t rope_dim, double rope_theta,
    void* workspace, size_t workspace_bytes,
    uint32_t* d_status, kvrp_stream_t stream);

/*
 * kv_relocate_batch_noalloc -- kv_relocate_batch for callers that cannot
 * allocate device memory.  The pages have no counterpart of this call; it
 * exists for integration.  Some callers own no device allocator at all: a
 * plugin inside a host engine that hands out only its own tensors, or a
 * serving process whose memory pool reserved all of the GPU up front, so that
 * an extra cudaMalloc either fails or breaks the pool's accounting; others
 * cannot afford the device-wide synchronisation an allocation may cause.
 * This call takes the same chunks and does the same work in the same single
 * kernel launch, but keeps the launch's descriptors in a fixed array inside
 * the library instead of a caller workspace (small copy kernels write them
 * there from their parameters).  It calls no cudaMalloc, cudaFree,
 * cudaHostAlloc or other allocating routine.
 *   Limits: at most KVRP_NOALLOC_MAX_CHUNKS chunks; more is rejected with
 *   KVRP_ERR_INVALID_ARG before any work.  The array (about 0.55 MB) lives on
 *   every GPU that loads the library, until the process exits.
 *   Set-up: the first call on a device looks up the array's device address
 *   with cudaGetSymbolAddress (the device must be current); make that first
 *   call before any stream capture.
 *   Sharing: every call on a device uses the same array, and each call
 *   rewrites the part its kernel reads.  Calls on one stream are ordered and
 *   safe; calls that can overlap on the GPU (different streams, or several
 *   host threads) race on the array and must not be issued.
 */
#define KVRP_NOALLOC_MAX_CHUNKS 256

kvrp_status kv_relocate_batch_noalloc(
    const kvrp_chunk* chunks, int32_t n_chunks,
    int32_t n_layers, int32_t n_kv_heads, int32_t head_dim, double rope_theta,
    uint32_t* d_status, kvrp_stream_t stream);

/*
 * Patch formation -- the rank-m factors of the conditioning deficit (Kamera,
 * section 2, patch bullet: computed once, at compile time or on first reuse,
 * from one conditioned pass over [A, B] followed by an SVD that keeps the
 * top-m factors).  The conditioned pass itself belongs to the model and is
 * the caller's: this call takes its output KV(B|A) together with the
 * canonical KV(B|empty) of the same tensor and forms
 *     Delta = KV(B|A) - R(delta) KV(B|empty)      (the destination frame)
 * per layer, then factors U_m [T][m] (singular values folded in) and
 * V_m [D][m] in bf16 such that U_m V_m^T approximates Delta, ready for
 * kv_relocate_patch / _mla / _batch.  The factorisation is a randomized range
 * finder with `power_iters` power iterations, Cholesky-QR orthonormalisation
 * and an fp32 Jacobi eigensolver on the small projected problem.
 *   conditioned, canonical  device bf16 [n_layers][n_tokens][row_width], rows
 *               dense; layer l at base + l * *_layer_stride elements (0: dense
 *               layers).  Only read.
 *   rope_kind   KVRP_ROPE_HEADS: every head of rot_dim features turns (keys;
 *               row_width a multiple of rot_dim);
 *               KVRP_ROPE_NONE: nothing turns (values; rot_dim, delta, theta unused);
 *               KVRP_ROPE_MLA_TAIL: the last rot_dim features turn (MLA k_rope).
 *               rot_dim: a multiple of 4, at most 128.  row_width: a multiple of 4.
 *   delta, rope_theta  the position shift and the RoPE base, as in kv_relocate_patch.
 *   rank, oversample  m >= 1 and the range finder's extra columns p >= 0;
 *               m + p <= 96, m <= min(n_tokens, row_width).
 *   power_iters 0..8 subspace iterations (1-2 suffice for decaying spectra).
 *   omega       device fp32 [row_width][m + p], row-major: the caller's Gaussian
 *               test matrix (N(0, 1) entries), shared by all layers; only read.
 *   u_out, v_out  device bf16 U_m [L][T][m] and V_m [L][row_width][m],
 *               row-major, layer strides u/v_layer_stride elements (0: dense);
 *               V_m has orthonormal columns, U_m = Delta V_m.
 *   workspace   device scratch of at least kv_patch_form_workspace_size(...)
 *               bytes, owned by the caller, busy until the call's work on
 *               `stream` completes (no two overlapping calls may share it).
 *               Calls with their own workspaces may run concurrently on
 *               different streams (K and V of one chunk, say): the k x k
 *               solves occupy one CTA per layer, so a second call's passes
 *               fill the rest of the GPU meanwhile.
 *   d_status    optional device word; KVRP_DEV_TIMEOUT is OR-ed in if a
 *               pipeline wait of the tensor-core passes gave up (results invalid).
 * Base pointers must be 16-byte aligned.  Precision: Delta is stored in bf16
 * (rows and transposed rows), the passes over it are bf16 x bf16 tensor-core
 * products accumulated in fp32; Gram matrices, the k x k solves (shifted
 * Cholesky QR, Jacobi) and the small products run in fp32; factors are rounded
 * once to bf16.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (sizes beyond the limits above)
 * and WORKSPACE are returned before any CUDA work is queued; CUDA if a launch
 * fails.  Asynchronous on `stream`; the result is an approximation of the
 * truncated SVD whose quality grows with p and power_iters.
 */
#define KVRP_ROPE_NONE 0
#define KVRP_ROPE_HEADS 1
#define KVRP_ROPE_MLA_TAIL 2

size_t kv_patch_form_workspace_size(int32_t n_layers, int32_t n_tokens, int32_t row_width,
                                    int32_t rank, int32_t oversample);

kvrp_status kv_patch_form(
    const void* conditioned, const void* canonical,
    int64_t cond_layer_stride, int64_t canon_layer_stride,
    int32_t n_layers, int32_t n_tokens, int32_t row_width,
    int32_t rope_kind, int32_t rot_dim, int64_t delta, double rope_theta,
    int32_t rank, int32_t oversample, int32_t power_iters, const float* omega,
    void* u_out, void* v_out, int64_t u_layer_stride, int64_t v_layer_stride,
    void* workspace, size_t workspace_bytes, uint32_t* d_status, kvrp_stream_t stream);

/*
 * Orbit patch (Kamera, section 3, reordering bullet: one patch, averaged over
 * the orderings of a cached set, serves every ordering).  Same as
 * kv_patch_form, with n_orbit conditioned caches KV(B|A_pi), each in its own
 * destination frame delta_pi, and the deficit averaged before the factorisation:
 *     Delta = (1/n) sum_pi [KV(B|A_pi) - R(delta_pi) KV(B|empty)].
 *   conditioned  host array of n_orbit device pointers (bf16, layout and
 *                layer stride as `conditioned` of kv_patch_form), only read.
 *   deltas       host array of the n_orbit position shifts.
 *   n_orbit      1..64 (UNSUPPORTED beyond).  n_orbit = 1 is kv_patch_form.
 * Other arguments, errors and precision as kv_patch_form.
 */
kvrp_status kv_patch_form_orbit(
    const void* const* conditioned, const int64_t* deltas, int32_t n_orbit,
    const void* canonical, int64_t cond_layer_stride, int64_t canon_layer_stride,
    int32_t n_layers, int32_t n_tokens, int32_t row_width,
    int32_t rope_kind, int32_t rot_dim, double rope_theta,
    int32_t rank, int32_t oversample, int32_t power_iters, const float* omega,
    void* u_out, void* v_out, int64_t u_layer_stride, int64_t v_layer_stride,
    void* workspace, size_t workspace_bytes, uint32_t* d_status, kvrp_stream_t stream);

/*
 * Decode attention over relocated, patched chunks, without writing the
 * relocated cache (the fused read-side use of the operator of Kamera, section 2:
 * a chunk cached as KV(B|empty) is read as K^ = R(delta) K + U_k V_k^T and
 * V^ = V + U_v V_v^T).  For one new query token per sequence,
 *     out[s][j] = softmax(softmax_scale * q[s][j] . K^_s) V^_s
 * over the concatenated chunks of sequence s, query head j reading KV head
 * j / (n_q_heads / n_kv_heads).  The query is rotated by R(-delta) once per
 * chunk and the key patch enters as (V_k^T q) . u_k,t, so a token costs its
 * canonical k_t, v_t and the rank-m rows u_k,t, u_v,t.
 *   q           device bf16 [n_seqs][n_q_heads][head_dim].
 *   chunks      host array of n_chunks (1..KVRP_ATTN_MAX_CHUNKS) kvrp_attn_chunk,
 *               ordered by sequence: sequence s owns chunks
 *               [seq_chunks[s], seq_chunks[s + 1]) (host array of n_seqs + 1,
 *               from 0 to n_chunks, non-decreasing).
 *   kvrp_attn_chunk.k, .v   device bf16 [n_tokens][n_kv_heads * head_dim] rows
 *               of one layer, or, with .block_table, pools [num_pages][16][row]
 *               in which token t of the chunk sits at page block_table[t / 16],
 *               slot t % 16 (a paged cache; an entry outside [0, num_pages)
 *               sets KVRP_DEV_BAD_PAGE and reads page 0 instead, the output then
 *               being undefined); .rank 0 or a multiple of 16 up to 128; .uk, .uv
 *               [n_tokens][rank], .vk, .vv [n_kv_heads * head_dim][rank] bf16
 *               (all four, or none when rank is 0); .delta the shift.
 *   head_dim    64 or 128; n_q_heads a multiple of n_kv_heads, at most 16x.
 *   out         device bf16 [n_seqs][n_q_heads][head_dim]; a sequence with no
 *               tokens gets zeros.
 *   workspace   device scratch of kv_attend_relocated_workspace_size(...) bytes
 *               (fp32 partial results and which blocks hold them); its contents
 *               need not survive between calls.  The size depends on the current
 *               device's SM count, and the call returns WORKSPACE if it is smaller
 *               than the size for the device it runs on.
 *   d_status    optional device word; KVRP_DEV_TIMEOUT is OR-ed in if an internal
 *               pipeline wait gave up (the output is then undefined).
 * Pointers 16-byte aligned.  Arithmetic fp32 on the bf16 inputs (rotation
 * angles in fp64; q, V_k^T q and the softmax weights enter the tensor-core
 * products as high + low bf16 parts), output rounded once to bf16.  Errors
 * (INVALID_ARG, ALIGNMENT, UNSUPPORTED -- also beyond 2^31 - 1 tokens in one
 * call -- and WORKSPACE) are returned before any CUDA work; CUDA on a launch
 * failure.  Asynchronous on `stream`.
 */
#define KVRP_ATTN_MAX_CHUNKS 256

typedef struct {
  const void* k;
  const void* v;
  int32_t n_tokens;
  int32_t rank;
  int64_t delta;
  const void* uk;
  const void* vk;
  const void* uv;
  const void* vv;
  const int32_t* block_table;  /* device; NULL => k, v are contiguous [n_tokens][row] */
  int32_t num_pages;           /* pages of the pool k, v point to (when block_table != NULL) */
} kvrp_attn_chunk;

size_t kv_attend_relocated_workspace_size(int32_t n_chunks, const int32_t* chunk_tokens, int32_t n_q_heads,
                                          int32_t n_kv_heads, int32_t head_dim);

kvrp_status kv_attend_relocated(
    const void* q, const kvrp_attn_chunk* chunks, int32_t n_chunks, const int32_t* seq_chunks,
    int32_t n_seqs, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
    double rope_theta, float softmax_scale, void* out,
    void* workspace, size_t workspace_bytes, uint32_t* d_status, kvrp_stream_t stream);

/*
 * kvrp_test_set_wait_limit -- for tests of the failure path only.  Sets the
 * limit, in SM clock cycles, of the relocation kernel's pipeline waits in the
 * plans built from now on by any thread (0 restores the default of about one
 * second).  With a limit of a few hundred cycles the waits give up almost at
 * once: the launch then ORs KVRP_DEV_TIMEOUT into *d_status, lets its copies
 * and tensor-core work drain, frees its TMEM and returns, leaving the output
 * incomplete.  It never hangs the GPU, whatever the limit.
 */
void kvrp_test_set_wait_limit(uint32_t cycles);

/*
 * kvrp_test_attend_split -- for tests of the host-side planning only; no CUDA
 * call.  The work split kv_attend_relocated gives n_cta blocks for chunks of
 * these token counts and ranks (host arrays of n_chunks): the stage sequence
 * (head group, chunk, stage) cut into contiguous shares of about equal bytes,
 * counting each stage's K, V and factor rows and each segment's V_k, query and
 * V_v slots.  Writes the boundaries share0[0 .. count] (share0 holds n_cta + 1
 * entries) and returns count (<= n_cta, every share non-empty), 0 when no chunk
 * has tokens, -1 on an invalid argument.  The other arguments are those of
 * kv_attend_relocated.
 */
int32_t kvrp_test_attend_split(const int32_t* chunk_tokens, const int32_t* chunk_ranks, int32_t n_chunks,
                               int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t n_cta,
                               int32_t* share0);

/* Human-readable name of a status code (static string). */
const char* kvrp_status_string(kvrp_status status);

/* Text of the last error seen by this host thread (static per thread). */
const char* kvrp_last_error(void);

/* Kernel launches that this host thread's last relocation call (kv_relocate_*)
 * or attention call (kv_attend_relocated) enqueued.  Relocation: the relocation
 * kernel, plus for a batch the small copy launches that carry its launch plan to
 * the device (31 KB of plan each).  Attention: the block and combine kernels (2;
 * the combine alone when no chunk has tokens).  0 when the call returned an
 * error or had nothing to move. */
int32_t kvrp_last_launch_count(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t kvrp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVRP_H */
