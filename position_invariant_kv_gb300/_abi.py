"""ctypes declarations of include/kvrp.h and thin wrappers with the same names."""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libkvrp.so")

KVRP_OK = 0
KVRP_ERR_INVALID_ARG = 1
KVRP_ERR_ALIGNMENT = 2
KVRP_ERR_UNSUPPORTED = 3
KVRP_ERR_CUDA = 4
KVRP_ERR_WORKSPACE = 5
KVRP_DEV_BAD_PAGE = 0x1
KVRP_DEV_TIMEOUT = 0x2

EXPORTED_SYMBOLS = (
    "kv_relocate_patch", "kv_relocate_patch_mrope", "kv_relocate_patch_mla", "kv_relocate_batch",
    "kv_relocate_batch_workspace_size", "kv_relocate_batch_noalloc", "kv_relocate_batch_mrope",
    "kv_relocate_batch_mla", "kvrp_test_set_wait_limit", "kvrp_test_attend_split", "kv_patch_form_workspace_size",
    "kv_patch_form", "kv_patch_form_orbit", "kv_attend_relocated_workspace_size", "kv_attend_relocated",
    "kvrp_status_string",
    "kvrp_last_error", "kvrp_last_launch_count", "kvrp_version",
)
KVRP_NOALLOC_MAX_CHUNKS = 256
KVRP_ROPE_NONE = 0
KVRP_ROPE_HEADS = 1
KVRP_ROPE_MLA_TAIL = 2


KVRP_ATTN_MAX_CHUNKS = 256


class kvrp_attn_chunk(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("n_tokens", C.c_int32), ("rank", C.c_int32),
                ("delta", C.c_int64), ("uk", C.c_void_p), ("vk", C.c_void_p), ("uv", C.c_void_p),
                ("vv", C.c_void_p), ("block_table", C.c_void_p), ("num_pages", C.c_int32)]


class kvrp_dst(C.Structure):
    _fields_ = [("base", C.c_void_p), ("layer_stride", C.c_int64), ("block_table", C.c_void_p),
                ("num_pages", C.c_int32), ("page_size", C.c_int32), ("dst_start", C.c_int64)]


class kvrp_chunk(C.Structure):
    _fields_ = [("k_src", C.c_void_p), ("v_src", C.c_void_p), ("src_layer_stride", C.c_int64),
                ("n_tokens", C.c_int32), ("rank", C.c_int32), ("delta", C.c_int64),
                ("uk", C.c_void_p), ("vk", C.c_void_p), ("uv", C.c_void_p), ("vv", C.c_void_p),
                ("u_layer_stride", C.c_int64), ("v_layer_stride", C.c_int64),
                ("k_dst", kvrp_dst), ("v_dst", kvrp_dst)]


class kvrp_mla_chunk(C.Structure):
    _fields_ = [("src", C.c_void_p), ("src_layer_stride", C.c_int64), ("n_tokens", C.c_int32),
                ("rank", C.c_int32), ("delta", C.c_int64), ("u", C.c_void_p), ("v", C.c_void_p),
                ("u_layer_stride", C.c_int64), ("v_layer_stride", C.c_int64), ("dst", kvrp_dst)]


def _load_library():
    if not os.path.exists(lib_path):
        raise ImportError(
            f"libkvrp.so is not built ({lib_path}); run `python -m position_invariant_kv_gb300.build` "
            "(there is no fallback implementation)")
    L = C.CDLL(lib_path)
    st = C.c_int
    L.kv_relocate_patch.restype = st
    L.kv_relocate_patch.argtypes = [
        C.c_void_p, C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
        C.c_int64, C.c_double, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
        C.c_int64, C.c_int64, C.POINTER(kvrp_dst), C.POINTER(kvrp_dst), C.c_void_p, C.c_void_p]
    L.kv_relocate_patch_mrope.restype = st
    L.kv_relocate_patch_mrope.argtypes = [
        C.c_void_p, C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
        C.POINTER(C.c_int64), C.POINTER(C.c_int32), C.c_double, C.c_int32, C.c_void_p, C.c_void_p,
        C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.POINTER(kvrp_dst), C.POINTER(kvrp_dst), C.c_void_p,
        C.c_void_p]
    L.kv_relocate_patch_mla.restype = st
    L.kv_relocate_patch_mla.argtypes = [
        C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int64, C.c_double,
        C.c_int32, C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.POINTER(kvrp_dst), C.c_void_p,
        C.c_void_p]
    L.kv_relocate_batch_workspace_size.restype = C.c_size_t
    L.kv_relocate_batch_workspace_size.argtypes = [C.c_int32]
    L.kv_relocate_batch.restype = st
    L.kv_relocate_batch.argtypes = [
        C.POINTER(kvrp_chunk), C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_double,
        C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p]
    L.kv_relocate_batch_mrope.restype = st
    L.kv_relocate_batch_mrope.argtypes = [
        C.POINTER(kvrp_chunk), C.POINTER(C.c_int64), C.c_int32, C.c_int32, C.c_int32, C.c_int32,
        C.POINTER(C.c_int32), C.c_double, C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p]
    L.kv_relocate_batch_mla.restype = st
    L.kv_relocate_batch_mla.argtypes = [
        C.POINTER(kvrp_mla_chunk), C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_double,
        C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p]
    L.kvrp_test_set_wait_limit.restype = None
    L.kvrp_test_set_wait_limit.argtypes = [C.c_uint32]
    L.kvrp_test_attend_split.restype = C.c_int32
    L.kvrp_test_attend_split.argtypes = [C.POINTER(C.c_int32), C.POINTER(C.c_int32), C.c_int32, C.c_int32,
                                         C.c_int32, C.c_int32, C.c_int32, C.POINTER(C.c_int32)]
    L.kv_relocate_batch_noalloc.restype = st
    L.kv_relocate_batch_noalloc.argtypes = [
        C.POINTER(kvrp_chunk), C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_double, C.c_void_p,
        C.c_void_p]
    L.kv_patch_form_workspace_size.restype = C.c_size_t
    L.kv_patch_form_workspace_size.argtypes = [C.c_int32] * 5
    L.kv_patch_form.restype = st
    L.kv_patch_form.argtypes = [
        C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
        C.c_int64, C.c_double, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
        C.c_int64, C.c_int64, C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p]
    L.kv_patch_form_orbit.restype = st
    L.kv_patch_form_orbit.argtypes = [
        C.POINTER(C.c_void_p), C.POINTER(C.c_int64), C.c_int32, C.c_void_p, C.c_int64, C.c_int64, C.c_int32,
        C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_double, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
        C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p]
    L.kv_attend_relocated_workspace_size.restype = C.c_size_t
    L.kv_attend_relocated_workspace_size.argtypes = [C.c_int32, C.POINTER(C.c_int32), C.c_int32, C.c_int32, C.c_int32]
    L.kv_attend_relocated.restype = st
    L.kv_attend_relocated.argtypes = [
        C.c_void_p, C.POINTER(kvrp_attn_chunk), C.c_int32, C.POINTER(C.c_int32), C.c_int32, C.c_int32, C.c_int32,
        C.c_int32, C.c_double, C.c_float, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p]
    L.kvrp_status_string.restype = C.c_char_p
    L.kvrp_status_string.argtypes = [C.c_int]
    L.kvrp_last_error.restype = C.c_char_p
    L.kvrp_last_error.argtypes = []
    L.kvrp_last_launch_count.restype = C.c_int32
    L.kvrp_last_launch_count.argtypes = []
    L.kvrp_version.restype = C.c_int32
    L.kvrp_version.argtypes = []
    return L


_LIB = None


def lib():
    """The loaded libkvrp.so.  Raises ImportError when it has not been built:
    there is no other implementation to fall back to."""
    global _LIB
    if _LIB is None:
        _LIB = _load_library()
    return _LIB


class KvrpError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        msg = lib().kvrp_status_string(status).decode()
        detail = lib().kvrp_last_error().decode()
        super().__init__(f"{msg}: {detail}" if detail else msg)


def kvrp_status_string(status: int) -> str:
    return lib().kvrp_status_string(status).decode()


def kvrp_last_launch_count() -> int:
    """Kernel launches of this thread's last relocation call (1 + plan-upload copies for a batch)."""
    return int(lib().kvrp_last_launch_count())


def kvrp_version() -> int:
    return int(lib().kvrp_version())


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int):
    if status != KVRP_OK:
        raise KvrpError(status)


@dataclass
class Dst:
    """One destination pool: layer l at base + l * layer_stride elements, laid
    out [num_pages][16][D]; block_table None means contiguous rows."""
    base: object
    num_pages: int
    layer_stride: int = 0
    block_table: object = None
    dst_start: int = 0
    page_size: int = 16

    def c(self) -> kvrp_dst:
        return kvrp_dst(_ptr(self.base), int(self.layer_stride), _ptr(self.block_table),
                        int(self.num_pages), int(self.page_size), int(self.dst_start))


@dataclass
class Chunk:
    """One chunk of kv_relocate_batch (fields as in struct kvrp_chunk)."""
    k_src: object
    v_src: object
    n_tokens: int
    delta: int
    k_dst: Dst
    v_dst: Dst
    rank: int = 0
    uk: object = None
    vk: object = None
    uv: object = None
    vv: object = None
    src_layer_stride: int = 0
    u_layer_stride: int = 0
    v_layer_stride: int = 0

    def c(self) -> kvrp_chunk:
        return kvrp_chunk(_ptr(self.k_src), _ptr(self.v_src), int(self.src_layer_stride),
                          int(self.n_tokens), int(self.rank), int(self.delta),
                          _ptr(self.uk), _ptr(self.vk), _ptr(self.uv), _ptr(self.vv),
                          int(self.u_layer_stride), int(self.v_layer_stride),
                          self.k_dst.c(), self.v_dst.c())


def kv_relocate_patch(k_src, v_src, *, n_layers: int, n_tokens: int, n_kv_heads: int, head_dim: int,
                      delta: int, rope_theta: float, k_dst: Dst, v_dst: Dst, rank: int = 0,
                      uk=None, vk=None, uv=None, vv=None, src_layer_stride: int = 0,
                      u_layer_stride: int = 0, v_layer_stride: int = 0, d_status=None,
                      stream=None) -> None:
    kd, vd = k_dst.c(), v_dst.c()
    _check(lib().kv_relocate_patch(
        _ptr(k_src), _ptr(v_src), int(src_layer_stride), int(n_layers), int(n_tokens), int(n_kv_heads),
        int(head_dim), int(delta), float(rope_theta), int(rank), _ptr(uk), _ptr(vk), _ptr(uv), _ptr(vv),
        int(u_layer_stride), int(v_layer_stride), C.byref(kd), C.byref(vd), _ptr(d_status),
        _stream(stream)))


def kv_relocate_patch_mrope(k_src, v_src, *, n_layers: int, n_tokens: int, n_kv_heads: int, head_dim: int,
                            delta_thw, mrope_section, rope_theta: float, k_dst: Dst, v_dst: Dst, rank: int = 0,
                            uk=None, vk=None, uv=None, vv=None, src_layer_stride: int = 0,
                            u_layer_stride: int = 0, v_layer_stride: int = 0, d_status=None,
                            stream=None) -> None:
    kd, vd = k_dst.c(), v_dst.c()
    d3 = (C.c_int64 * 3)(*[int(v) for v in delta_thw])
    s3 = (C.c_int32 * 3)(*[int(v) for v in mrope_section])
    _check(lib().kv_relocate_patch_mrope(
        _ptr(k_src), _ptr(v_src), int(src_layer_stride), int(n_layers), int(n_tokens), int(n_kv_heads),
        int(head_dim), d3, s3, float(rope_theta), int(rank), _ptr(uk), _ptr(vk), _ptr(uv), _ptr(vv),
        int(u_layer_stride), int(v_layer_stride), C.byref(kd), C.byref(vd), _ptr(d_status), _stream(stream)))


def kv_relocate_patch_mla(src, *, n_layers: int, n_tokens: int, kv_lora_dim: int, rope_dim: int,
                          delta: int, rope_theta: float, dst: Dst, rank: int = 0, u=None, v=None,
                          src_layer_stride: int = 0, u_layer_stride: int = 0, v_layer_stride: int = 0,
                          d_status=None, stream=None) -> None:
    d = dst.c()
    _check(lib().kv_relocate_patch_mla(
        _ptr(src), int(src_layer_stride), int(n_layers), int(n_tokens), int(kv_lora_dim), int(rope_dim),
        int(delta), float(rope_theta), int(rank), _ptr(u), _ptr(v), int(u_layer_stride),
        int(v_layer_stride), C.byref(d), _ptr(d_status), _stream(stream)))


def kv_relocate_batch_workspace_size(n_chunks: int) -> int:
    return int(lib().kv_relocate_batch_workspace_size(int(n_chunks)))


def chunk_array(chunks: Sequence[Chunk]):
    """The ctypes array of struct kvrp_chunk for a list of chunks.  Build it once
    and pass it to the batch calls when the same chunks are relocated again."""
    return (kvrp_chunk * max(1, len(chunks)))(*[c.c() for c in chunks])


def _as_array(chunks):
    if isinstance(chunks, C.Array):
        return chunks, len(chunks)
    return chunk_array(chunks), len(chunks)


def kv_relocate_batch(chunks, *, n_layers: int, n_kv_heads: int, head_dim: int,
                      rope_theta: float, workspace, workspace_bytes: Optional[int] = None,
                      d_status=None, stream=None) -> None:
    """chunks: a list of Chunk, or an array made by chunk_array()."""
    arr, n = _as_array(chunks)
    if workspace_bytes is None:
        workspace_bytes = int(workspace.numel() * workspace.element_size())
    _check(lib().kv_relocate_batch(
        arr, n, int(n_layers), int(n_kv_heads), int(head_dim), float(rope_theta),
        _ptr(workspace), int(workspace_bytes), _ptr(d_status), _stream(stream)))


def kv_relocate_batch_mrope(chunks, delta_thw, *, n_layers: int, n_kv_heads: int, head_dim: int,
                            mrope_section, rope_theta: float, workspace, workspace_bytes: Optional[int] = None,
                            d_status=None, stream=None) -> None:
    """kv_relocate_batch under M-RoPE: chunk i turns by the (t, h, w) shift delta_thw[i]."""
    arr, n = _as_array(chunks)
    if len(delta_thw) != n:
        raise ValueError("one (t, h, w) shift per chunk")
    d = (C.c_int64 * max(3 * n, 3))(*[int(v) for t in delta_thw for v in t])
    s3 = (C.c_int32 * 3)(*[int(v) for v in mrope_section])
    if workspace_bytes is None:
        workspace_bytes = int(workspace.numel() * workspace.element_size())
    _check(lib().kv_relocate_batch_mrope(
        arr, d, n, int(n_layers), int(n_kv_heads), int(head_dim), s3, float(rope_theta),
        _ptr(workspace), int(workspace_bytes), _ptr(d_status), _stream(stream)))


@dataclass
class MlaChunk:
    """One chunk of kv_relocate_batch_mla (fields as in struct kvrp_mla_chunk)."""
    src: object
    n_tokens: int
    delta: int
    dst: Dst
    rank: int = 0
    u: object = None
    v: object = None
    src_layer_stride: int = 0
    u_layer_stride: int = 0
    v_layer_stride: int = 0

    def c(self) -> kvrp_mla_chunk:
        return kvrp_mla_chunk(_ptr(self.src), int(self.src_layer_stride), int(self.n_tokens), int(self.rank),
                              int(self.delta), _ptr(self.u), _ptr(self.v), int(self.u_layer_stride),
                              int(self.v_layer_stride), self.dst.c())


def mla_chunk_array(chunks: Sequence[MlaChunk]):
    """The ctypes array of struct kvrp_mla_chunk for a list of MLA chunks."""
    return (kvrp_mla_chunk * max(1, len(chunks)))(*[c.c() for c in chunks])


def kv_relocate_batch_mla(chunks, *, n_layers: int, kv_lora_dim: int, rope_dim: int, rope_theta: float,
                          workspace, workspace_bytes: Optional[int] = None, d_status=None, stream=None) -> None:
    """Many MLA chunks, each with its own delta and patch, in one launch.
    chunks: a list of MlaChunk, or an array made by mla_chunk_array()."""
    if isinstance(chunks, C.Array):
        arr, n = chunks, len(chunks)
    else:
        arr, n = mla_chunk_array(chunks), len(chunks)
    if workspace_bytes is None:
        workspace_bytes = int(workspace.numel() * workspace.element_size())
    _check(lib().kv_relocate_batch_mla(
        arr, n, int(n_layers), int(kv_lora_dim), int(rope_dim), float(rope_theta), _ptr(workspace),
        int(workspace_bytes), _ptr(d_status), _stream(stream)))


def kvrp_test_set_wait_limit(cycles: int) -> None:
    """Testing hook: the relocation kernel's pipeline wait limit in cycles for
    plans built from now on (0 = the default, about one second)."""
    lib().kvrp_test_set_wait_limit(int(cycles))


def kvrp_test_attend_split(tokens, ranks, *, n_q_heads: int, n_kv_heads: int, head_dim: int, n_cta: int):
    """Testing hook: the share boundaries kv_attend_relocated would give n_cta
    blocks for chunks of these token counts and ranks (a list of count + 1
    stage indices), [] when no chunk has tokens; ValueError on invalid input."""
    n = len(tokens)
    t = (C.c_int32 * n)(*[int(x) for x in tokens])
    r = (C.c_int32 * n)(*[int(x) for x in ranks])
    out = (C.c_int32 * (int(n_cta) + 1))()
    cnt = lib().kvrp_test_attend_split(t, r, n, int(n_q_heads), int(n_kv_heads), int(head_dim), int(n_cta), out)
    if cnt < 0:
        raise ValueError("kvrp_test_attend_split: invalid arguments")
    return [out[i] for i in range(cnt + 1)] if cnt > 0 else []


def kv_relocate_batch_noalloc(chunks, *, n_layers: int, n_kv_heads: int, head_dim: int,
                              rope_theta: float, d_status=None, stream=None) -> None:
    """kv_relocate_batch without a workspace, for callers that cannot allocate
    device memory: the launch descriptors go to a fixed array inside the
    library (at most KVRP_NOALLOC_MAX_CHUNKS chunks; calls that can overlap on
    the GPU must not be issued, as they share that array)."""
    arr, n = _as_array(chunks)
    _check(lib().kv_relocate_batch_noalloc(
        arr, n, int(n_layers), int(n_kv_heads), int(head_dim), float(rope_theta),
        _ptr(d_status), _stream(stream)))


def kv_patch_form_workspace_size(n_layers: int, n_tokens: int, row_width: int, rank: int, oversample: int) -> int:
    return int(lib().kv_patch_form_workspace_size(int(n_layers), int(n_tokens), int(row_width), int(rank),
                                                  int(oversample)))


def kv_patch_form(conditioned, canonical, *, n_layers: int, n_tokens: int, row_width: int, rope_kind: int,
                  rot_dim: int, delta: int, rope_theta: float, rank: int, oversample: int, power_iters: int,
                  omega, u_out, v_out, workspace, cond_layer_stride: int = 0, canon_layer_stride: int = 0,
                  u_layer_stride: int = 0, v_layer_stride: int = 0, workspace_bytes: Optional[int] = None,
                  d_status=None, stream=None) -> None:
    """Rank-m factors of Delta = conditioned - R(delta) canonical, per layer (bf16 U_m, V_m)."""
    if workspace_bytes is None:
        workspace_bytes = int(workspace.numel() * workspace.element_size())
    _check(lib().kv_patch_form(
        _ptr(conditioned), _ptr(canonical), int(cond_layer_stride), int(canon_layer_stride), int(n_layers),
        int(n_tokens), int(row_width), int(rope_kind), int(rot_dim), int(delta), float(rope_theta), int(rank),
        int(oversample), int(power_iters), _ptr(omega), _ptr(u_out), _ptr(v_out), int(u_layer_stride),
        int(v_layer_stride), _ptr(workspace), int(workspace_bytes), _ptr(d_status), _stream(stream)))


def kv_patch_form_orbit(conditioned, deltas, canonical, *, n_layers: int, n_tokens: int, row_width: int,
                        rope_kind: int, rot_dim: int, rope_theta: float, rank: int, oversample: int,
                        power_iters: int, omega, u_out, v_out, workspace, cond_layer_stride: int = 0,
                        canon_layer_stride: int = 0, u_layer_stride: int = 0, v_layer_stride: int = 0,
                        workspace_bytes: Optional[int] = None, d_status=None, stream=None) -> None:
    """Orbit patch: factors of mean_pi [conditioned_pi - R(delta_pi) canonical], per layer."""
    n = len(conditioned)
    if len(deltas) != n:
        raise ValueError("one delta per conditioned cache")
    ptrs = (C.c_void_p * max(n, 1))(*[_ptr(c) for c in conditioned])
    ds = (C.c_int64 * max(n, 1))(*[int(d) for d in deltas])
    if workspace_bytes is None:
        workspace_bytes = int(workspace.numel() * workspace.element_size())
    _check(lib().kv_patch_form_orbit(
        ptrs, ds, n, _ptr(canonical), int(cond_layer_stride), int(canon_layer_stride), int(n_layers),
        int(n_tokens), int(row_width), int(rope_kind), int(rot_dim), float(rope_theta), int(rank),
        int(oversample), int(power_iters), _ptr(omega), _ptr(u_out), _ptr(v_out), int(u_layer_stride),
        int(v_layer_stride), _ptr(workspace), int(workspace_bytes), _ptr(d_status), _stream(stream)))


@dataclass
class AttnChunk:
    """One chunk of kv_attend_relocated (fields as in struct kvrp_attn_chunk)."""
    k: object
    v: object
    n_tokens: int
    delta: int = 0
    rank: int = 0
    uk: object = None
    vk: object = None
    uv: object = None
    vv: object = None
    block_table: object = None   # int32 device tensor: page of each 16 tokens (None: contiguous rows)
    num_pages: int = 0

    def c(self) -> kvrp_attn_chunk:
        return kvrp_attn_chunk(_ptr(self.k), _ptr(self.v), int(self.n_tokens), int(self.rank), int(self.delta),
                               _ptr(self.uk), _ptr(self.vk), _ptr(self.uv), _ptr(self.vv),
                               _ptr(self.block_table), int(self.num_pages))


def kv_attend_relocated_workspace_size(chunk_tokens, n_q_heads: int, n_kv_heads: int, head_dim: int) -> int:
    """Scratch bytes of kv_attend_relocated (depends on the current device's SM count)."""
    n = len(chunk_tokens)
    arr = (C.c_int32 * max(n, 1))(*[int(t) for t in chunk_tokens])
    return int(lib().kv_attend_relocated_workspace_size(n, arr, int(n_q_heads), int(n_kv_heads), int(head_dim)))


def attn_chunk_array(chunks):
    """ctypes array of kvrp_attn_chunk for kv_attend_relocated (reusable across calls)."""
    arr = (kvrp_attn_chunk * max(len(chunks), 1))()
    for i, c in enumerate(chunks):
        arr[i] = c.c()
    return arr, len(chunks)


def kv_attend_relocated(q, chunks, seq_chunks, *, n_q_heads: int, n_kv_heads: int, head_dim: int, rope_theta: float,
                        softmax_scale: float, out, workspace, workspace_bytes: Optional[int] = None,
                        d_status=None, stream=None) -> None:
    """Decode attention of one query token per sequence over relocated, patched chunks."""
    arr, n = chunks if isinstance(chunks, tuple) else attn_chunk_array(chunks)
    sc = (C.c_int32 * len(seq_chunks))(*[int(v) for v in seq_chunks])
    if workspace_bytes is None:
        workspace_bytes = int(workspace.numel() * workspace.element_size())
    _check(lib().kv_attend_relocated(
        _ptr(q), arr, n, sc, len(seq_chunks) - 1, int(n_q_heads), int(n_kv_heads), int(head_dim), float(rope_theta),
        float(softmax_scale), _ptr(out), _ptr(workspace), int(workspace_bytes), _ptr(d_status), _stream(stream)))
