"""fp64 CPU oracle for the Kamera KV reuse operator.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import or call it.  It shares no code with the CUDA path
(``position_invariant_kv_gb300``): no kernels, headers, tables, constants or
pre/post-processing.  Its only common dependency with that path is the seeded
input generator module ``workloads``, which holds none of the method's
arithmetic.

What it computes (Kamera, gist.science/pt/paper/2606.23581, section 2 "O
Operador Kamera"; the Korean summary gist.science/ko/paper/2606.23581 section 2
states the same):

    KV^(B|A) = R(delta) . KV(B|empty) + U_m V_m^T

* ``R(delta)`` re-rotates cached keys by the RoPE phase of the position shift
  delta; it is an exact algebraic operation, not a forward pass.
* ``U_m V_m^T`` is a rank-m conditioning patch, added after the relocation.
* GQA/MHA: full keys are relocated, values are not rotated, both are patched.
* MLA: only the decoupled 64-dim k_rope is relocated, c_KV is reused byte for
  byte, and the patch is added to both channels.

Everything is computed in fp64 from the bf16 inputs and rounded once,
nearest-even, to bf16.  Pins for every function live in ``tests/test_oracle_*``
(closed forms, group laws, SVD brute force, exhaustive bf16 checks, a
hand-derived golden example).  Parity of the whole operator at workload scale
beyond those pins is unpinned: the pages print no worked numeric example.
"""
from .bf16 import bf16_bits_to_f64, round_to_bf16_bits, bf16_ord, ulp_distance, bf16_ulp
from .kamera import (
    inv_freq, rope_absolute, mrope_absolute, pair_shifts, relocate, patch_product, row_layout, operator_rows,
    conditioning, placement, run_workload, chunk_layer_rows,
)
from .patch_svd import svd_patch, eckart_young_tail, conditioning_deficit, orbit_deficit
from .attend import attention, attend_relocated, attend_conditioning, relocated_chunk

__all__ = [
    "bf16_bits_to_f64", "round_to_bf16_bits", "bf16_ord", "ulp_distance", "bf16_ulp",
    "inv_freq", "rope_absolute", "mrope_absolute", "pair_shifts", "relocate", "patch_product", "row_layout", "operator_rows",
    "conditioning", "placement", "run_workload", "chunk_layer_rows",
    "svd_patch", "eckart_young_tail", "conditioning_deficit", "orbit_deficit",
    "attention", "attend_relocated", "attend_conditioning", "relocated_chunk",
]
