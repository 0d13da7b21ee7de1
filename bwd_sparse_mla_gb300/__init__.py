"""GB300 (sm_103a) sparse MLA attention: forward and backward through a C ABI.

Importing the package loads nothing; `bwd_sparse_mla_gb300.capi` loads the
in-tree libsparse_mla.so on first use and fails loudly if it is missing.
"""
__all__ = ["capi", "workloads", "build"]
