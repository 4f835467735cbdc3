"""Python binding of libkvrp, the GB300 KV relocation + rank-m patch library.

Argument marshalling only: every step of the operator runs in the library's
CUDA kernel.  Names mirror the C ABI in include/kvrp.h:

    kv_relocate_patch        GQA/MHA chunk, all layers, K and V
    kv_relocate_patch_mrope  the same under M-RoPE (per-section temporal/height/width shifts)
    kv_relocate_patch_mla    MLA chunk (c_KV ++ k_rope rows)
    kv_relocate_batch        many GQA/MHA chunks, each with its own delta and patch
    kv_relocate_batch_mrope  the same under M-RoPE, each chunk with its own (t, h, w) shift
    kv_relocate_batch_mla    many MLA chunks, each with its own delta and patch
    kv_relocate_batch_noalloc  kv_relocate_batch without a workspace (fixed in-library array)
    kv_relocate_batch_workspace_size
    kv_patch_form            rank-m factors of the conditioning deficit (patch formation)
    kv_patch_form_orbit      the same, deficit averaged over the orderings of a cached set
    kv_attend_relocated      decode attention over relocated, patched chunks (never materialised)

Tensors may be passed as torch CUDA tensors (their data_ptr is used) or as raw
device addresses (int).  Streams default to torch's current stream.  A status
other than KVRP_OK raises KvrpError.  There is no CPU fallback: importing the
package fails when libkvrp.so has not been built.
"""
from __future__ import annotations

from ._abi import (  # noqa: F401
    KVRP_DEV_BAD_PAGE, KVRP_DEV_TIMEOUT, KVRP_OK, KVRP_ERR_INVALID_ARG, KVRP_ERR_ALIGNMENT,
    KVRP_ERR_UNSUPPORTED, KVRP_ERR_CUDA, KVRP_ERR_WORKSPACE,
    Dst, Chunk, KvrpError, lib, lib_path,
    kv_relocate_patch, kv_relocate_patch_mrope, kv_relocate_patch_mla, kv_relocate_batch, kv_relocate_batch_workspace_size,
    kvrp_status_string, kvrp_version, kvrp_last_launch_count, EXPORTED_SYMBOLS,
    kv_relocate_batch_noalloc, KVRP_NOALLOC_MAX_CHUNKS, chunk_array,
    kv_relocate_batch_mrope, kv_relocate_batch_mla, MlaChunk, mla_chunk_array, kvrp_test_set_wait_limit,
    kvrp_test_attend_split,
    kv_patch_form, kv_patch_form_orbit, kv_patch_form_workspace_size,
    kv_attend_relocated, kv_attend_relocated_workspace_size, AttnChunk, attn_chunk_array, KVRP_ATTN_MAX_CHUNKS,
    KVRP_ROPE_NONE, KVRP_ROPE_HEADS, KVRP_ROPE_MLA_TAIL,
)
