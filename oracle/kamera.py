"""The Kamera reuse operator in plain fp64 (oracle; test infrastructure only).

Source: Kamera, gist.science/pt/paper/2606.23581, section 2 "O Operador Kamera"
(reuse equation, relocation bullet, patch bullet, the MHA / GQA / MLA family
bullets), mirrored by gist.science/ko/paper/2606.23581 section 2; the
composable-KV section 3.B of gist.science/pt/paper/2606.17107 ("Models take
notes in prefill") confirms that keys are re-rotated to their new absolute
positions while values, being position-free, are transplanted unchanged.

Readings of points the pages leave open:
  * RoPE is the rotate-half convention: feature i of a rotated head pairs with
    feature i + d/2; the pair turns by phi_i = delta * theta_i with
    theta_i = theta_base ** (-2 i / d), i = 0 .. d/2 - 1, all in fp64.
  * delta is the new position minus the old one, one value per chunk, so
    R(delta) . RoPE(k, p) = RoPE(k, p + delta).
  * M-RoPE (the multimodal RoPE of Qwen-VL-style models, whose image KV is
    re-rotated by M-RoPE in the composable-KV summary, section 4): the
    frequency pairs form consecutive temporal / height / width sections and
    delta is a (d_t, d_h, d_w) tuple, pair i turning by its section's shift.
  * The patch is added after the rotation and is not itself rotated (the
    reuse equation read literally).
  * K and V each carry their own factor pair (U [T][m], W [D][m]); MLA carries
    one pair over the whole 576-wide row.
  * Destination pages hold 16 tokens; the block table maps logical page
    (position // 16) of a sequence to a physical page; a contiguous
    destination is the identity table.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_bits_to_f64, round_to_bf16_bits

PAGE = 16


# --------------------------------------------------------------------------- #
# R(delta): exact RoPE re-rotation (Kamera section 2, relocation bullet)
# --------------------------------------------------------------------------- #

def inv_freq(rot_dim: int, theta: float) -> np.ndarray:
    """theta_i = theta ** (-2 i / rot_dim) for i = 0 .. rot_dim/2 - 1 (fp64)."""
    i = np.arange(rot_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / rot_dim)


def _turn(x: np.ndarray, phi: np.ndarray) -> np.ndarray:
    """Turn each rotate-half pair (x_i, x_{i+h}) of the last axis by phi_i."""
    h = x.shape[-1] // 2
    x1, x2 = x[..., :h], x[..., h:]
    c, s = np.cos(phi), np.sin(phi)
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_absolute(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """RoPE of rows x [n][d] at absolute positions pos [n] (the encoding a model
    applies at prefill).  Used only to pin R(delta)."""
    x = np.asarray(x, dtype=np.float64)
    phi = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq(x.shape[-1], theta)[None, :]
    return _turn(x, phi)


def pair_shifts(delta, n_pairs: int, sections=None) -> np.ndarray:
    """Position shift seen by each frequency pair.  Plain RoPE: every pair
    shifts by delta.  M-RoPE (multimodal RoPE of Qwen-VL-style models): the
    frequency pairs are split into consecutive (temporal, height, width)
    sections, and pair i shifts by the component of delta = (d_t, d_h, d_w)
    that owns its section."""
    if sections is None:
        return np.full(n_pairs, np.float64(delta))
    assert sum(sections) == n_pairs, "sections must cover every frequency pair"
    return np.repeat(np.asarray(delta, dtype=np.float64), np.asarray(sections))


def relocate(x: np.ndarray, delta, theta: float, sections=None) -> np.ndarray:
    """R(delta) applied to rows whose last axis is one rotated head; with
    M-RoPE sections, delta is the (t, h, w) shift tuple."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    phi = pair_shifts(delta, d // 2, sections) * inv_freq(d, theta)
    return _turn(x, phi)


def mrope_absolute(x: np.ndarray, pos_thw: np.ndarray, theta: float, sections) -> np.ndarray:
    """M-RoPE of rows x [n][d] at 3-component positions pos_thw [n][3] (the
    encoding a multimodal model applies at prefill).  Used only to pin R(delta)."""
    x = np.asarray(x, dtype=np.float64)
    pos = np.repeat(np.asarray(pos_thw, dtype=np.float64), np.asarray(sections), axis=1)
    phi = pos * inv_freq(x.shape[-1], theta)[None, :]
    return _turn(x, phi)


# --------------------------------------------------------------------------- #
# Row layout per family (Kamera section 2, "Suporte a Arquitetura Unificada")
# --------------------------------------------------------------------------- #

def row_layout(family: str, tensor: str, *, n_heads=0, head_dim=0, kv_lora_dim=0, rope_dim=0):
    """Segments (start, width, rotated) of one token row.

    gqa/mha keys: every head is rotated; values: nothing is rotated;
    mla: c_KV [0, kv_lora_dim) untouched, k_rope [kv_lora_dim, +rope_dim) rotated."""
    if family == "mla":
        return [(0, kv_lora_dim, False), (kv_lora_dim, rope_dim, True)]
    D = n_heads * head_dim
    if tensor == "k":
        return [(h * head_dim, head_dim, True) for h in range(n_heads)]
    return [(0, D, False)]


def _layout_of(wl, tensor):
    return row_layout(wl.family, tensor, n_heads=wl.n_heads, head_dim=wl.head_dim,
                      kv_lora_dim=wl.kv_lora_dim, rope_dim=wl.rope_dim)


def apply_relocation(x: np.ndarray, delta, theta: float, layout, sections=None) -> np.ndarray:
    """R(delta) on rows [n][D] following a row layout."""
    y = np.array(x, dtype=np.float64, copy=True)
    for start, width, rotated in layout:
        if rotated:
            y[:, start:start + width] = relocate(y[:, start:start + width], delta, theta, sections)
    return y


# --------------------------------------------------------------------------- #
# The rank-m patch (Kamera section 2, patch bullet)
# --------------------------------------------------------------------------- #

def patch_product(u_bits, w_bits) -> np.ndarray:
    """U_m V_m^T in fp64 from bf16 factors U [n][m] and W [D][m].  Each product
    of two bf16 values is exact in fp64."""
    u = bf16_bits_to_f64(u_bits)
    w = bf16_bits_to_f64(w_bits)
    return u @ w.T


# --------------------------------------------------------------------------- #
# The operator on a block of rows
# --------------------------------------------------------------------------- #

def operator_rows(x_bits, u_bits, w_bits, delta, theta, layout, sections=None) -> np.ndarray:
    """fp64 value of R(delta) x + U W^T for rows x [n][D] (bf16 bits)."""
    y = apply_relocation(bf16_bits_to_f64(x_bits), delta, theta, layout, sections)
    if u_bits is not None:
        y = y + patch_product(u_bits, w_bits)
    return y


def conditioning(x_bits, u_bits, w_bits, delta, theta, layout, sections=None) -> np.ndarray:
    """Sum of magnitudes of the terms that make up each output element:
    |x_i cos| + |x_j sin| for a rotated element (|x| otherwise) plus
    sum_r |U_tr W_fr|.  Rounding errors of any evaluation order are bounded by
    a small multiple of unit roundoff times this sum."""
    x = np.abs(bf16_bits_to_f64(x_bits))
    s = np.array(x, copy=True)
    for start, width, rotated in layout:
        if not rotated:
            continue
        h = width // 2
        phi = pair_shifts(delta, h, sections) * inv_freq(width, theta)
        c, sn = np.abs(np.cos(phi)), np.abs(np.sin(phi))
        x1 = x[:, start:start + h]
        x2 = x[:, start + h:start + width]
        s[:, start:start + h] = x1 * c + x2 * sn
        s[:, start + h:start + width] = x2 * c + x1 * sn
    if u_bits is not None:
        s = s + np.abs(bf16_bits_to_f64(u_bits)) @ np.abs(bf16_bits_to_f64(w_bits)).T
    return s


# --------------------------------------------------------------------------- #
# Paged placement (block table of 16-token pages)
# --------------------------------------------------------------------------- #

def placement(wl, chunk):
    """(page, slot) of every token of a chunk, by a plain loop over tokens:
    position q = dst_start + t, logical page q // 16, slot q % 16, physical page
    from the sequence's block table (identity when the destination is contiguous)."""
    pages = np.empty(chunk.n_tokens, dtype=np.int64)
    slots = np.empty(chunk.n_tokens, dtype=np.int64)
    for t in range(chunk.n_tokens):
        q = chunk.dst_start + t
        logical = q // PAGE
        if wl.paged:
            pages[t] = int(wl.block_tables[chunk.seq][logical])
        else:
            pages[t] = logical
        slots[t] = q % PAGE
    return pages, slots


def chunk_layer_rows(wl, inputs, ci: int, tensor: str, layer: int, tokens=None):
    """(ref fp64 [n][D], conditioning [n][D]) for chosen tokens of one chunk,
    layer and tensor.  ``inputs`` holds host uint16 arrays (see workloads)."""
    c = wl.chunks[ci]
    tok = np.arange(c.n_tokens) if tokens is None else np.asarray(tokens)
    x = inputs["rows"][tensor][layer, c.src_row0 + tok]
    u = w = None
    if c.rank:
        u = inputs["u"][tensor][ci][layer, tok]
        w = inputs["w"][tensor][ci][layer]
    lay = _layout_of(wl, tensor)
    sec = getattr(wl, "mrope_sections", None)
    ref = operator_rows(x, u, w, c.delta, wl.theta, lay, sec)
    cond = conditioning(x, u, w, c.delta, wl.theta, lay, sec)
    return ref, cond


def run_workload(wl, inputs, sentinel=0xFFFF):
    """Whole destination pools after every chunk of a (small) workload has been
    relocated, patched, rounded to bf16 and placed.  Untargeted slots keep the
    sentinel bit pattern.  Returns ({tensor: uint16 [L][pages][16][D]},
    {tensor: fp64 ref pools}, {tensor: fp64 conditioning pools})."""
    L, D = wl.n_layers, wl.row_width
    pools, refs, conds = {}, {}, {}
    for name in wl.tensors:
        pool = np.full((L, wl.num_pages, PAGE, D), sentinel, dtype=np.uint16)
        refp = np.full((L, wl.num_pages, PAGE, D), np.nan)
        condp = np.zeros((L, wl.num_pages, PAGE, D))
        for ci, c in enumerate(wl.chunks):
            pages, slots = placement(wl, c)
            for l in range(L):
                ref, cond = chunk_layer_rows(wl, inputs, ci, name, l)
                pool[l, pages, slots] = round_to_bf16_bits(ref)
                refp[l, pages, slots] = ref
                condp[l, pages, slots] = cond
        pools[name], refs[name], conds[name] = pool, refp, condp
    return pools, refs, conds
