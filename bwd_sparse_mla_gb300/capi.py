"""Thin ctypes binding of libsparse_mla.so (argument marshalling only).

Function names match the C ABI in include/sparse_mla.h.  Tensors are torch
CUDA tensors (PyTorch supplies device memory and streams); every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or the call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsparse_mla.so")

SMLA_DKV_ATOMIC = 0
SMLA_DKV_DETERMINISTIC = 1
D_QK = 576
D_V = 512

_lib = None


class SparseMLAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"sparse_mla error {code}: {msg}")
        self.code = code


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with bwd_sparse_mla_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.sparse_mla_fwd.argtypes = [P, P, P, P, I, I, I, I, F, P, P, P]
    lib.sparse_mla_fwd.restype = I
    lib.sparse_mla_fwd_rows.argtypes = [P, P, P, P, I, I, I, I, F, I, I, P, P, P]
    lib.sparse_mla_fwd_rows.restype = I
    lib.sparse_mla_bwd_rows.argtypes = [P, P, P, P, P, P, P, I, I, I, I, F, I, I, P, P, P, S, P]
    lib.sparse_mla_bwd_rows.restype = I
    lib.sparse_mla_dkv_cast.argtypes = [P, P, I, P]
    lib.sparse_mla_dkv_cast.restype = I
    lib.sparse_mla_bwd_workspace_bytes.argtypes = [I, I, I, I]
    lib.sparse_mla_bwd_workspace_bytes.restype = S
    lib.sparse_mla_bwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, F, I, P, P, P, P, S, P]
    lib.sparse_mla_bwd.restype = I
    lib.sparse_mla_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, F, P, P, P, P]
    lib.sparse_mla_bwd_noalloc.restype = I
    lib.sparse_mla_check_indices.argtypes = [P, I, I, P, I, ctypes.POINTER(ctypes.c_int64), P]
    lib.sparse_mla_check_indices.restype = I
    lib.sparse_mla_last_error.argtypes = []
    lib.sparse_mla_last_error.restype = ctypes.c_char_p
    lib.sparse_mla_version.argtypes = []
    lib.sparse_mla_version.restype = ctypes.c_char_p
    lib.sparse_mla_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), I]
    lib.sparse_mla_device_status.restype = I
    lib.sparse_mla_launch_count.argtypes = []
    lib.sparse_mla_launch_count.restype = ctypes.c_uint64
    lib.sparse_mla_wait_selftest.argtypes = [P]
    lib.sparse_mla_wait_selftest.restype = I
    lib.sparse_mla_bounds_selftest.argtypes = [P]
    lib.sparse_mla_bounds_selftest.restype = I
    lib.sparse_mla_topk.argtypes = [P, ctypes.c_int64, I, I, P, I, I, P, P]
    lib.sparse_mla_topk.restype = I
    _lib = lib
    return lib


def sparse_mla_last_error() -> str:
    return load().sparse_mla_last_error().decode()


def sparse_mla_version() -> str:
    return load().sparse_mla_version().decode()


def sparse_mla_launch_count() -> int:
    return int(load().sparse_mla_launch_count())


def sparse_mla_device_status(clear: bool = False) -> int:
    st = ctypes.c_uint32(0)
    _check(load().sparse_mla_device_status(ctypes.byref(st), int(clear)))
    return int(st.value)


def sparse_mla_wait_selftest(stream=None) -> None:
    """Enqueue the bounded-wait self-test: a wait that nothing releases gives
    up after 1 s and sets the device status word to 1 (read and clear it with
    sparse_mla_device_status(clear=True))."""
    _check(load().sparse_mla_wait_selftest(_stream(stream)))


def sparse_mla_bounds_selftest(stream=None) -> None:
    """Debug build only (-DSMLA_DEBUG): enqueue the bounds-check self-test; both of
    its probes fall outside their buffer, so the device status word becomes 2.  The
    product build refuses it (-ENOSYS)."""
    _check(load().sparse_mla_bounds_selftest(_stream(stream)))


def sparse_mla_topk(scores, cu_seqlens, topk: int, ncols: int | None = None, indices=None, stream=None):
    """indices [T, 1, topk] int32: per row the best min(topk, causal count) candidates
    of scores [T, ncols] (fp32, row-major) as packed kv rows, -1 padded."""
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be a row-major [T, ncols] float32 tensor")
    T = scores.shape[0]
    ncols = scores.shape[1] if ncols is None else int(ncols)
    if indices is None:
        indices = torch.empty((T, 1, topk), dtype=torch.int32, device=scores.device)
    _check(load().sparse_mla_topk(_ptr(scores), scores.stride(0), T, ncols, _ptr(cu_seqlens), cu_seqlens.numel() - 1,
                                  int(topk), _ptr(indices), _stream(stream)))
    return indices


def _check(rc: int) -> None:
    if rc != 0:
        raise SparseMLAError(rc, sparse_mla_last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dims(q, indices):
    T, H, dq = q.shape
    assert dq == D_QK, "q must be [T, H, 576]"
    topk = indices.shape[-1]
    return T, H, topk


def sparse_mla_fwd(q, kv, indices, cu_seqlens, scale, out=None, lse=None, stream=None):
    """out [T,H,512] bf16, lse [T,H] fp32 = forward of q [T,H,576] bf16,
    kv [T,1,576] bf16, indices [T,1,topk] int32 (-1 = padding)."""
    T, H, topk = _dims(q, indices)
    if out is None:
        out = torch.empty((T, H, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check(load().sparse_mla_fwd(_ptr(q), _ptr(kv), _ptr(indices), _ptr(cu_seqlens), T, H, topk, B,
                                 float(scale), _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def sparse_mla_fwd_rows(q, kv, indices, cu_seqlens, scale, t0: int, nt: int, out, lse, stream=None):
    """Forward of query rows [t0, t0 + nt) into the full out [T,H,512] / lse [T,H]
    (the other rows are neither read nor written)."""
    T, H, topk = _dims(q, indices)
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check(load().sparse_mla_fwd_rows(_ptr(q), _ptr(kv), _ptr(indices), _ptr(cu_seqlens), T, H, topk, B,
                                      float(scale), int(t0), int(nt), _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def sparse_mla_bwd_rows(q, kv, out, dout, lse, indices, cu_seqlens, scale, t0: int, nt: int, dq, dkv_f32,
                        workspace, stream=None):
    """Backward of query rows [t0, t0 + nt): writes those rows of dq and ADDS their
    dKV contributions into dkv_f32 (zeroed by the caller before the first range)."""
    T, H, topk = _dims(q, indices)
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check(load().sparse_mla_bwd_rows(_ptr(q), _ptr(kv), _ptr(out), _ptr(dout), _ptr(lse), _ptr(indices),
                                      _ptr(cu_seqlens), T, H, topk, B, float(scale), int(t0), int(nt), _ptr(dq),
                                      _ptr(dkv_f32), _ptr(workspace), workspace.numel(), _stream(stream)))
    return dq, dkv_f32


def sparse_mla_dkv_cast(dkv_f32, dkv, stream=None):
    """dkv (bf16) = round-to-nearest-even of dkv_f32 [T,1,576]."""
    _check(load().sparse_mla_dkv_cast(_ptr(dkv_f32), _ptr(dkv), dkv_f32.shape[0], _stream(stream)))
    return dkv


def sparse_mla_bwd_workspace_bytes(T: int, H: int, topk: int, dkv_mode: int = SMLA_DKV_ATOMIC) -> int:
    return int(load().sparse_mla_bwd_workspace_bytes(T, H, topk, dkv_mode))


def sparse_mla_bwd(q, kv, out, dout, lse, indices, cu_seqlens, scale, dkv_mode=SMLA_DKV_ATOMIC,
                   dq=None, dkv_f32=None, dkv=None, workspace=None, want_bf16_dkv=True, stream=None):
    """dq [T,H,576] bf16, dkv_f32 [T,1,576] fp32 and (optionally) dkv bf16."""
    T, H, topk = _dims(q, indices)
    dev = q.device
    if dq is None:
        dq = torch.empty((T, H, D_QK), dtype=torch.bfloat16, device=dev)
    if dkv_f32 is None:
        dkv_f32 = torch.empty((T, 1, D_QK), dtype=torch.float32, device=dev)
    if dkv is None and want_bf16_dkv:
        dkv = torch.empty((T, 1, D_QK), dtype=torch.bfloat16, device=dev)
    need = sparse_mla_bwd_workspace_bytes(T, H, topk, dkv_mode)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check(load().sparse_mla_bwd(_ptr(q), _ptr(kv), _ptr(out), _ptr(dout), _ptr(lse), _ptr(indices),
                                 _ptr(cu_seqlens), T, H, topk, B, float(scale), int(dkv_mode), _ptr(dq),
                                 _ptr(dkv_f32), _ptr(dkv), _ptr(workspace), workspace.numel(),
                                 _stream(stream)))
    return dq, dkv_f32, dkv


NOALLOC_MAX_ROWS = 1 << 23   # T * H limit of sparse_mla_bwd_noalloc


def sparse_mla_bwd_noalloc(q, kv, out, dout, lse, indices, cu_seqlens, scale, dq=None, dkv_f32=None,
                           dkv=None, want_bf16_dkv=True, stream=None):
    """Backward that needs no workspace (the library keeps Delta in a fixed
    device array, T*H <= 2^23).  Calls that overlap on the GPU race on that
    array.  Output tensors may be passed in so that nothing is allocated."""
    T, H, topk = _dims(q, indices)
    dev = q.device
    if dq is None:
        dq = torch.empty((T, H, D_QK), dtype=torch.bfloat16, device=dev)
    if dkv_f32 is None:
        dkv_f32 = torch.empty((T, 1, D_QK), dtype=torch.float32, device=dev)
    if dkv is None and want_bf16_dkv:
        dkv = torch.empty((T, 1, D_QK), dtype=torch.bfloat16, device=dev)
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check(load().sparse_mla_bwd_noalloc(_ptr(q), _ptr(kv), _ptr(out), _ptr(dout), _ptr(lse), _ptr(indices),
                                         _ptr(cu_seqlens), T, H, topk, B, float(scale), _ptr(dq),
                                         _ptr(dkv_f32), _ptr(dkv), _stream(stream)))
    return dq, dkv_f32, dkv


def sparse_mla_check_indices(indices, cu_seqlens, stream=None) -> int:
    T = indices.shape[0]
    topk = indices.shape[-1]
    B = cu_seqlens.numel() - 1
    n_bad = ctypes.c_int64(0)
    _check(load().sparse_mla_check_indices(_ptr(indices), T, topk, _ptr(cu_seqlens), B,
                                           ctypes.byref(n_bad), _stream(stream)))
    return int(n_bad.value)
