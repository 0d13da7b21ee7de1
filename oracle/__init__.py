"""fp64 CPU oracle for sparse MLA attention -- test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
"""
from .sparse_mla_ref import (  # noqa: F401
    D_LATENT, D_QK, D_TAIL, LSE_EMPTY, SUMEXP_FLOOR, bf16_bits_to_f64, check_indices, delta,
    sparse_mla_bwd, sparse_mla_fwd, valid_slots,
)
