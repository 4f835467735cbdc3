"""The parity rule that decides whether a bf16 result agrees with the fp64 oracle
(test infrastructure only).

An element passes when its bf16 value is within 1 bf16 ulp of the oracle
rounded to bf16.  A rotated element whose exact value nearly cancels (|ref|
far below the magnitudes of the terms that form it) can legitimately be
further away in ulps of its own tiny value; such an element is still
accepted, and counted as a mismatch, when the absolute error stays within
one ulp of ref plus 2^-20 times the conditioning sum (|x_i cos| + |x_j sin| +
sum_r |U_tr V_fr|).  Any element outside that bound is a violation.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_bits_to_f64, round_to_bf16_bits, ulp_distance, bf16_ulp

COND_FACTOR = 2.0 ** -20


def parity_report(got_bits, ref, cond) -> dict:
    got_bits = np.asarray(got_bits, dtype=np.uint16).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    cond = np.asarray(cond, dtype=np.float64).ravel()
    want = round_to_bf16_bits(ref)
    d = ulp_distance(got_bits, want)
    g = bf16_bits_to_f64(got_bits)
    err = np.abs(g - ref)
    bound = bf16_ulp(ref) + COND_FACTOR * cond
    mism = d > 1
    viol = mism & ~(err <= bound)
    nz = ref != 0
    rel = float(np.max(err[nz] / np.abs(ref[nz]))) if nz.any() else 0.0
    rel_ok = err[~mism & nz] / np.abs(ref[~mism & nz]) if nz.any() else np.zeros(0)
    return {
        "n": int(d.size),
        "ulp0": int(np.sum(d == 0)),
        "ulp1": int(np.sum(d == 1)),
        "mismatches": int(np.sum(mism)),
        "violations": int(np.sum(viol)),
        "max_ulp": int(d.max()) if d.size else 0,
        "max_rel_err": rel,
        "max_rel_err_within_1ulp": float(rel_ok.max()) if rel_ok.size else 0.0,
    }
