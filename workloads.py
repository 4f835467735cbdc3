"""Seeded synthetic workloads for the KV relocation + rank-m patch operator.

This module only draws inputs: canonical K/V rows, patch factors, position
shifts and block tables.  It holds none of the operator's arithmetic (no
rotation, no patch product, no rounding of results), so that both the fp64
oracle and the CUDA path can consume the same inputs without sharing any of
the method's code.

Shapes and distributions follow the five workloads the operator is measured on
(video-segment GQA, reordered MHA chunks with an orbit patch, DeepSeek-style
MLA, and a sliding-window survival + recall batch), as described for the Kamera
operator (gist.science/pt/paper/2606.23581, section 2 "O Operador Kamera" and
section 3 "Tres Operacoes de Janela Baratas").

Recipe (stated once, used everywhere):
  * canonical rows: x[l, t, f] = z * s[l, tensor, f], z ~ N(0, 1) per element,
    s ~ lognormal(mean=0, sigma=0.5) per feature channel, drawn per layer and
    per tensor (K, V), then rounded to bf16;
  * patch factors: U [L][T][m] and W [L][D][m], entries N(0, std=0.05), bf16;
  * block tables: shuffled permutations of the physical pages (int32);
  * shifts: integers drawn inclusively from the stated ranges.

Two backends draw the numbers:
  * ``numpy``: ``numpy.random.default_rng(seed)`` on the host; bit-stable
    across machines and numpy versions; used for every case small enough to
    generate on the host;
  * ``torch``: ``torch.Generator(device).manual_seed(seed)``; used for the
    multi-GB workloads where host generation would take minutes.  Values differ
    from the numpy backend but are fixed by (seed, device type).

bf16 data is carried as uint16 bit patterns on the host (numpy has no bf16).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

PAGE = 16  # tokens per destination page


@dataclass(frozen=True)
class Chunk:
    """One cached chunk to be relocated into the destination cache."""

    src_row0: int    # first row of the chunk in the canonical store (per layer)
    n_tokens: int
    delta: object    # RoPE position shift (new - old); a (t, h, w) tuple under M-RoPE
    rank: int        # patch rank m (0 = relocation only)
    seq: int         # block-table row (paged destinations); 0 for contiguous
    dst_start: int   # first destination position of the chunk in its sequence


@dataclass
class Workload:
    name: str
    family: str              # "gqa" (also MHA when n_heads == query heads) or "mla"
    n_layers: int
    n_heads: int             # KV heads (gqa); 1 for mla
    head_dim: int            # gqa head dim; mla: rope dim
    kv_lora_dim: int         # mla: c_KV width; 0 for gqa
    rope_dim: int            # rotated width per head (gqa: head_dim; mla: 64)
    theta: float
    src_rows: int            # rows per layer of the canonical store
    num_pages: int           # destination pages per layer (contiguous: rows // 16)
    paged: bool
    chunks: list = field(default_factory=list)
    block_tables: Optional[np.ndarray] = None   # int32 [n_seq][pages_per_seq]
    seed: int = 0
    backend: str = "numpy"
    mrope_sections: Optional[tuple] = None   # (t, h, w) frequency-pair counts under M-RoPE

    @property
    def row_width(self) -> int:
        """Features per token row of one tensor (D)."""
        if self.family == "mla":
            return self.kv_lora_dim + self.rope_dim
        return self.n_heads * self.head_dim

    @property
    def tensors(self) -> tuple:
        return ("kv",) if self.family == "mla" else ("k", "v")

    @property
    def n_chunk_tokens(self) -> int:
        return sum(c.n_tokens for c in self.chunks)

    def algorithmic_bytes(self) -> dict:
        """Bytes the operator must move: canonical rows read, factors read,
        destination rows written (block tables and descriptors excluded)."""
        D = self.row_width
        nt = len(self.tensors)
        rows = self.n_chunk_tokens * self.n_layers * nt
        kv_read = rows * D * 2
        written = kv_read
        factors = 0
        for c in self.chunks:
            if c.rank:
                factors += self.n_layers * nt * (c.n_tokens + D) * c.rank * 2
        return {"kv_read": kv_read, "factors": factors, "written": written,
                "total": kv_read + factors + written}

    def patch_flops(self) -> int:
        D = self.row_width
        nt = len(self.tensors)
        return sum(2 * c.rank * c.n_tokens * D * self.n_layers * nt for c in self.chunks)


# --------------------------------------------------------------------------- #
# Workload descriptors
# --------------------------------------------------------------------------- #

def _perm_pages(rng, n):
    return rng.permutation(n).astype(np.int32)


def config(i: int, seed: Optional[int] = None) -> Workload:
    """The five measured workloads.  Seed defaults to 1000 + i."""
    seed = 1000 + i if seed is None else seed
    rng = np.random.default_rng(seed)
    if i == 0:
        # single chunk, 1 layer, GQA 8x128, delta +137, theta 1e6, m = 16, contiguous
        return Workload("c0_gqa_single", "gqa", 1, 8, 128, 0, 128, 1e6, 256, 256 // PAGE,
                        False, [Chunk(0, 256, 137, 16, 0, 0)], None, seed, "numpy")
    if i == 1:
        # Qwen2.5-VL-7B-shaped: 28 layers, 4 KV heads x 128, one 4096-token chunk
        delta = int(rng.integers(-32768, 32768, endpoint=True))
        bt = _perm_pages(rng, 4096 // PAGE)[None, :]
        return Workload("c1_qwen25vl_gqa", "gqa", 28, 4, 128, 0, 128, 1e6, 4096, 4096 // PAGE,
                        True, [Chunk(0, 4096, delta, 32, 0, 0)], bt, seed, "numpy")
    if i == 2:
        # Llama-2-7B-shaped MHA: 8 chunks of 2048 placed by a random permutation
        n, T = 8, 2048
        pi = rng.permutation(n)
        chunks = [Chunk(c * T, T, int(pi[c] - c) * T, 64, 0, int(pi[c]) * T) for c in range(n)]
        bt = _perm_pages(rng, n * T // PAGE)[None, :]
        return Workload("c2_llama2_mha_reorder", "gqa", 32, 32, 128, 0, 128, 1e4, n * T,
                        n * T // PAGE, True, chunks, bt, seed, "torch")
    if i == 3:
        # DeepSeek-V2-shaped MLA: 60 layers, 512 c_KV + 64 k_rope, 8192 tokens
        delta = int(rng.integers(-65536, 65536, endpoint=True))
        bt = _perm_pages(rng, 8192 // PAGE)[None, :]
        return Workload("c3_deepseekv2_mla", "mla", 60, 1, 64, 512, 64, 1e4, 8192, 8192 // PAGE,
                        True, [Chunk(0, 8192, delta, 32, 0, 0)], bt, seed, "torch")
    if i == 4:
        # sliding-window survival + recall: 8 requests x 32 chunks x 1024 tokens
        R, S, T = 8, 32, 1024
        pages_per_req = S * T // PAGE
        perm = _perm_pages(rng, R * pages_per_req)
        bt = perm.reshape(R, pages_per_req)
        chunks = []
        for r in range(R):
            recalled = set(int(s) for s in rng.choice(S, size=4, replace=False))
            for s in range(S):
                if s in recalled:
                    delta = int(rng.integers(-32768, 32768, endpoint=True))
                    rank = 64
                else:
                    delta = -int(rng.integers(1, 8, endpoint=True)) * T
                    rank = 0
                chunks.append(Chunk((r * S + s) * T, T, delta, rank, r, s * T))
        return Workload("c4_window_survive_recall", "gqa", 28, 4, 128, 0, 128, 1e6, R * S * T,
                        R * pages_per_req, True, chunks, bt, seed, "torch")
    if i == 5:
        # Qwen2.5-VL-shaped video segment under M-RoPE: 28 layers, 4 KV heads x 128,
        # frequency sections (16, 24, 24); the segment moves by a temporal shift and
        # a spatial base shift drawn independently
        dt = int(rng.integers(-32768, 32768, endpoint=True))
        ds = int(rng.integers(-32768, 32768, endpoint=True))
        bt = _perm_pages(rng, 4096 // PAGE)[None, :]
        return Workload("c5_qwen25vl_mrope", "gqa", 28, 4, 128, 0, 128, 1e6, 4096, 4096 // PAGE,
                        True, [Chunk(0, 4096, (dt, ds, ds), 32, 0, 0)], bt, seed, "numpy",
                        mrope_sections=(16, 24, 24))
    raise ValueError(f"no workload {i}")


def small_gqa(*, seed: int, n_layers=2, n_heads=2, head_dim=128, chunks_spec=((200, 37, 16, 0),),
              paged=True, theta=1e6, extra_pages=0, dst_starts=None, name="small_gqa",
              mrope_sections=None) -> Workload:
    """A host-sized GQA workload.  chunks_spec: (n_tokens, delta, rank, seq) per chunk.
    Destinations are packed one after another in each sequence unless dst_starts
    is given; pools get ``extra_pages`` unused pages so placement is checked."""
    rng = np.random.default_rng(seed)
    chunks, pos, row = [], {}, 0
    for k, (T, delta, rank, seq) in enumerate(chunks_spec):
        start = dst_starts[k] if dst_starts is not None else pos.get(seq, 0)
        chunks.append(Chunk(row, T, delta, rank, seq, start))
        pos[seq] = start + T
        row += T
    n_seq = max(c.seq for c in chunks) + 1
    pages_per_seq = max((c.dst_start + c.n_tokens + PAGE - 1) // PAGE for c in chunks)
    if paged:
        num_pages = n_seq * pages_per_seq + extra_pages
        bt = rng.permutation(num_pages)[: n_seq * pages_per_seq].astype(np.int32)
        bt = bt.reshape(n_seq, pages_per_seq)
    else:
        num_pages = pages_per_seq + extra_pages
        bt = None
    return Workload(name, "gqa", n_layers, n_heads, head_dim, 0, head_dim, theta, row, num_pages,
                    paged, chunks, bt, seed, "numpy", mrope_sections=mrope_sections)


def small_mla(*, seed: int, n_layers=2, n_tokens=150, delta=-999, rank=32, paged=True,
              dst_start=0, theta=1e4, kv_lora_dim=512, rope_dim=64, extra_pages=0, chunks_spec=None) -> Workload:
    """A host-sized MLA workload: one chunk (n_tokens, delta, rank at dst_start),
    or, with chunks_spec = ((n_tokens, delta, rank, seq), ...), several chunks
    packed one after another in each sequence."""
    rng = np.random.default_rng(seed)
    if chunks_spec is None:
        chunks_spec, starts = ((n_tokens, delta, rank, 0),), [dst_start]
    else:
        starts, pos = [], {}
        for T, _, _, seq in chunks_spec:
            starts.append(pos.get(seq, dst_start))
            pos[seq] = starts[-1] + T
    chunks, row = [], 0
    for (T, d, m, seq), start in zip(chunks_spec, starts):
        chunks.append(Chunk(row, T, d, m, seq, start))
        row += T
    n_seq = max(c.seq for c in chunks) + 1
    pages = max((c.dst_start + c.n_tokens + PAGE - 1) // PAGE for c in chunks)
    if paged:
        num_pages = n_seq * pages + extra_pages
        bt = rng.permutation(num_pages)[: n_seq * pages].astype(np.int32).reshape(n_seq, pages)
    else:
        num_pages, bt = pages + extra_pages, None
    return Workload("small_mla", "mla", n_layers, 1, rope_dim, kv_lora_dim, rope_dim, theta,
                    row, num_pages, paged, chunks, bt, seed, "numpy")


# --------------------------------------------------------------------------- #
# Drawing the numbers
# --------------------------------------------------------------------------- #

def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 draws to bf16 bit patterns (nearest-even).  Input
    generation only: the draws are finite and far from overflow."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def host_inputs(wl: Workload) -> dict:
    """Draw every input of a workload on the host (numpy backend).

    Returns uint16 (bf16 bit) arrays:
      rows[name]   [L][src_rows][D] for each tensor name in wl.tensors
      u[name][c]   [L][T_c][m_c] for patched chunks (None when m_c == 0)
      w[name][c]   [L][D][m_c]
    plus 'block_tables' (int32 or None)."""
    rng = np.random.default_rng(np.random.SeedSequence([wl.seed, 7]))
    L, D = wl.n_layers, wl.row_width
    rows = {}
    for name in wl.tensors:
        out = np.empty((L, wl.src_rows, D), np.uint16)
        for l in range(L):
            scale = rng.lognormal(0.0, 0.5, size=D)
            z = rng.standard_normal((wl.src_rows, D))
            out[l] = _f32_to_bf16_bits((z * scale).astype(np.float32))
        rows[name] = out
    u = {n: [] for n in wl.tensors}
    w = {n: [] for n in wl.tensors}
    for c in wl.chunks:
        for name in wl.tensors:
            if c.rank == 0:
                u[name].append(None)
                w[name].append(None)
                continue
            uu = rng.normal(0.0, 0.05, size=(L, c.n_tokens, c.rank)).astype(np.float32)
            ww = rng.normal(0.0, 0.05, size=(L, D, c.rank)).astype(np.float32)
            u[name].append(_f32_to_bf16_bits(uu))
            w[name].append(_f32_to_bf16_bits(ww))
    return {"rows": rows, "u": u, "w": w, "block_tables": wl.block_tables}


def torch_inputs(wl: Workload, device: str):
    """Draw every input of a workload with torch on ``device`` (torch backend).
    Returns bf16 tensors with the layouts of :func:`host_inputs`."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(wl.seed))
    L, D = wl.n_layers, wl.row_width
    rows = {}
    for name in wl.tensors:
        out = torch.empty((L, wl.src_rows, D), dtype=torch.bfloat16, device=device)
        for l in range(L):
            scale = torch.empty(D, dtype=torch.float32, device=device).log_normal_(0.0, 0.5, generator=g)
            z = torch.randn((wl.src_rows, D), dtype=torch.float32, device=device, generator=g)
            out[l] = (z * scale).to(torch.bfloat16)
            del z
        rows[name] = out
    u = {n: [] for n in wl.tensors}
    w = {n: [] for n in wl.tensors}
    for c in wl.chunks:
        for name in wl.tensors:
            if c.rank == 0:
                u[name].append(None)
                w[name].append(None)
                continue
            uu = torch.randn((L, c.n_tokens, c.rank), generator=g, device=device) * 0.05
            ww = torch.randn((L, D, c.rank), generator=g, device=device) * 0.05
            u[name].append(uu.to(torch.bfloat16))
            w[name].append(ww.to(torch.bfloat16))
    bt = None
    if wl.block_tables is not None:
        bt = torch.from_numpy(np.ascontiguousarray(wl.block_tables)).to(device)
    return {"rows": rows, "u": u, "w": w, "block_tables": bt}
