"""Patch formation by truncated SVD (oracle; test infrastructure only).

Kamera (gist.science/pt/paper/2606.23581, section 2, patch bullet) forms the
rank-m patch once: a conditioned pass over [A, B] gives KV(B|A), the deficit
Delta = KV(B|A) - KV(B|empty) is decomposed by an SVD, and the top-m factors
are kept.  The model pass is out of scope here; given a Delta, this module
returns the factors.  Reading: Delta is taken in the destination frame,
Delta = KV(B|A) - R(delta) KV(B|empty), so that adding U_m V_m^T after the
relocation reproduces KV(B|A); singular values are folded into U.
"""
from __future__ import annotations

import numpy as np


def svd_patch(delta_kv: np.ndarray, m: int):
    """(U_m [T][m], W_m [D][m]) with U_m W_m^T the best rank-m approximation of
    delta_kv in Frobenius norm; singular values are folded into U_m."""
    u, s, vt = np.linalg.svd(np.asarray(delta_kv, dtype=np.float64), full_matrices=False)
    return u[:, :m] * s[None, :m], vt[:m].T


def eckart_young_tail(delta_kv: np.ndarray, m: int) -> float:
    """Sum of the squared singular values beyond the first m."""
    s = np.linalg.svd(np.asarray(delta_kv, dtype=np.float64), compute_uv=False)
    return float(np.sum(s[m:] ** 2))


def conditioning_deficit(cond_rows: np.ndarray, canon_rows: np.ndarray, delta, theta: float, layout,
                         sections=None) -> np.ndarray:
    """Delta = KV(B|A) - R(delta) KV(B|empty) for rows [n][D] given in fp64
    (already decoded from bf16): the matrix whose top-m factors make the patch.
    R(delta) follows the row layout (keys: every head turned; values: none;
    MLA: only k_rope turned), exactly as the reuse operator applies it."""
    from .kamera import apply_relocation
    return np.asarray(cond_rows, dtype=np.float64) - apply_relocation(canon_rows, delta, theta, layout, sections)


def orbit_deficit(cond_rows_list, canon_rows: np.ndarray, deltas, theta: float, layout,
                  sections=None) -> np.ndarray:
    """Deficit of the orbit patch (Kamera, section 3, reordering bullet: one
    patch averaged over the orderings of a cached set): the mean over the
    orderings pi of KV(B|A_pi) - R(delta_pi) KV(B|empty), each deficit taken in
    its own destination frame delta_pi."""
    if len(cond_rows_list) != len(deltas) or not len(deltas):
        raise ValueError("one delta per conditioned cache, at least one")
    total = np.zeros(np.shape(canon_rows), dtype=np.float64)
    for cond_rows, delta in zip(cond_rows_list, deltas):
        total += conditioning_deficit(cond_rows, canon_rows, delta, theta, layout, sections)
    return total / len(deltas)
