"""Shared helpers of the GPU tests: moving seeded workloads to the device and
comparing CUDA results with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle.sparse_mla_ref as orc

# Tolerance stated for this path: relative Frobenius error <= 3e-3 (the
# figure the miles PR #2079 summary quotes for the fixed kernels against an
# fp32 reference) and max-abs error <= 2e-2, both against the fp64 oracle.
REL_FRO = 3e-3
MAX_ABS = 2e-2
LSE_EMPTY_F32 = np.float32(orc.LSE_EMPTY)


def bf16_dev(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def f64_to_bf16_dev(x: np.ndarray, dev) -> torch.Tensor:
    return torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).to(dev)


def device_inputs(w, dev):
    return dict(
        q=bf16_dev(w.q, dev),
        kv=bf16_dev(w.kv, dev),
        dout=bf16_dev(w.dout, dev),
        indices=torch.from_numpy(np.ascontiguousarray(w.indices)).to(dev),
        cu_seqlens=torch.from_numpy(w.cu_seqlens).to(dev),
    )


def err_stats(gpu: np.ndarray, ref: np.ndarray):
    diff = gpu - ref
    nref = np.linalg.norm(ref)
    rel = float(np.linalg.norm(diff) / nref) if nref > 0 else float(np.linalg.norm(diff))
    return rel, float(np.abs(diff).max()) if diff.size else 0.0


def assert_close(name: str, gpu: np.ndarray, ref: np.ndarray, rel_tol=REL_FRO, abs_tol=MAX_ABS):
    """rel_fro(gpu, ref) <= rel_tol, and |gpu - ref| <= abs_tol * max(1, |ref|)
    element by element.

    The max-abs bound is stated for unit-scale values.  A bf16 output of
    magnitude in [4, 8) is quantised in steps of 2^-5 = 0.031, so no bf16
    result can be within 2e-2 of fp64 there; above magnitude 1 the bound is
    therefore taken relative to the element's own magnitude."""
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    rel, mab = err_stats(gpu, ref)
    excess = np.abs(gpu - ref) / np.maximum(1.0, np.abs(ref)) if ref.size else np.zeros(1)
    worst = float(excess.max()) if excess.size else 0.0
    assert rel <= rel_tol and worst <= abs_tol, \
        f"{name}: rel_fro={rel:.3e} max_abs={mab:.3e} max_abs/max(1,|ref|)={worst:.3e}"
    return rel, mab


def empty_rows(w) -> np.ndarray:
    idx = w.indices.reshape(w.T, -1)
    return np.nonzero(~np.any((idx >= 0) & (idx < w.T), axis=1))[0]


def oracle_inputs(w):
    """q, kv, dout as f64 from the bf16 bits."""
    return (orc.bf16_bits_to_f64(w.q), orc.bf16_bits_to_f64(w.kv).reshape(w.T, -1),
            orc.bf16_bits_to_f64(w.dout))
