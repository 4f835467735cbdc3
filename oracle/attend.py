"""Decode attention over relocated, patched chunks (oracle; test infrastructure only).

The fused read-side use of the Kamera reuse operator (Kamera,
gist.science/pt/paper/2606.23581, section 2, "O Operador Kamera"): a new
query token attends to a context assembled from cached chunks, each stored in
its canonical form KV(B|empty) and reused at a new position with its shift
delta and rank-m patch,

    K^ = R(delta) K + U_k V_k^T,     V^ = V + U_v V_v^T,

without writing the relocated cache.  This module is the plain definition:
it materialises K^ and V^ of every chunk in fp64 (unrounded), concatenates the
chunks of a sequence, and evaluates softmax(scale q K^T) V^ per query head in
fp64, query head j reading KV head j // (n_q_heads / n_kv_heads) (grouped-query
attention).  The result is rounded once to bf16.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_bits_to_f64, round_to_bf16_bits
from .kamera import apply_relocation, patch_product, row_layout


def relocated_chunk(k_bits, v_bits, delta, theta: float, n_kv_heads: int, head_dim: int, uk=None, vk=None,
                    uv=None, vv=None, sections=None):
    """(K^, V^) of one chunk in fp64, [T][H_kv * d] each: the reuse operator
    before rounding."""
    lk = row_layout("gqa", "k", n_heads=n_kv_heads, head_dim=head_dim)
    lv = row_layout("gqa", "v", n_heads=n_kv_heads, head_dim=head_dim)
    k = apply_relocation(bf16_bits_to_f64(k_bits), delta, theta, lk, sections)
    v = apply_relocation(bf16_bits_to_f64(v_bits), delta, theta, lv, sections)
    if uk is not None:
        k = k + patch_product(uk, vk)
    if uv is not None:
        v = v + patch_product(uv, vv)
    return k, v


def attention(q, k, v, n_q_heads: int, n_kv_heads: int, head_dim: int, scale: float) -> np.ndarray:
    """softmax(scale q K^T) V for one query token: q [H_q * d], K and V
    [T][H_kv * d] (fp64); query head j reads KV head j // (H_q / H_kv).
    Returns [H_q * d] fp64."""
    g = n_q_heads // n_kv_heads
    q = np.asarray(q, dtype=np.float64).reshape(n_q_heads, head_dim)
    k = np.asarray(k, dtype=np.float64).reshape(-1, n_kv_heads, head_dim)
    v = np.asarray(v, dtype=np.float64).reshape(-1, n_kv_heads, head_dim)
    out = np.empty((n_q_heads, head_dim))
    for j in range(n_q_heads):
        h = j // g
        s = scale * (k[:, h, :] @ q[j])
        p = np.exp(s - s.max())
        out[j] = (p / p.sum()) @ v[:, h, :]
    return out.reshape(-1)


def attend_relocated(q_bits, chunks, n_q_heads: int, n_kv_heads: int, head_dim: int, theta: float, scale: float):
    """fp64 output [H_q * d] for one sequence.  `chunks` is a list of dicts
    with bf16 bits k, v [T][H_kv * d], delta, and optional uk, vk, uv, vv."""
    ks, vs = [], []
    for c in chunks:
        k, v = relocated_chunk(c["k"], c["v"], c["delta"], theta, n_kv_heads, head_dim, c.get("uk"), c.get("vk"),
                               c.get("uv"), c.get("vv"))
        ks.append(k)
        vs.append(v)
    return attention(bf16_bits_to_f64(q_bits), np.concatenate(ks), np.concatenate(vs), n_q_heads, n_kv_heads,
                     head_dim, scale)


def attend_conditioning(q_bits, chunks, n_q_heads: int, n_kv_heads: int, head_dim: int, theta: float,
                        scale: float) -> np.ndarray:
    """Sum over tokens of p_t |V^_t| per output element (the magnitude the
    output is assembled from); rounding errors of any evaluation order are a
    small multiple of unit roundoff times this sum."""
    g = n_q_heads // n_kv_heads
    ks, vs = [], []
    for c in chunks:
        k, v = relocated_chunk(c["k"], c["v"], c["delta"], theta, n_kv_heads, head_dim, c.get("uk"), c.get("vk"),
                               c.get("uv"), c.get("vv"))
        ks.append(k)
        vs.append(v)
    k = np.concatenate(ks).reshape(-1, n_kv_heads, head_dim)
    v = np.concatenate(vs).reshape(-1, n_kv_heads, head_dim)
    q = bf16_bits_to_f64(q_bits).reshape(n_q_heads, head_dim)
    out = np.empty((n_q_heads, head_dim))
    for j in range(n_q_heads):
        h = j // g
        s = scale * (k[:, h, :] @ q[j])
        p = np.exp(s - s.max())
        out[j] = (p / p.sum()) @ np.abs(v[:, h, :])
    return out.reshape(-1)


def round_output(x) -> np.ndarray:
    return round_to_bf16_bits(x)
