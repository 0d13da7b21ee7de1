"""Single-call dump and replay of a backward call.

The slime issue #2201 report ("Strongest repro evidence") debugs a bad
`sparse_mla_bwd(q, kv, tl_out, grad_output, indices, tl_lse, sm_scale)` call by
saving its inputs, re-running the call on them, counting the non-finite
entries of dq and dkv, and comparing against a reference on the finite
overlap.  This module saves such a call to one .npz file and re-runs the
library's backward on it; the comparison against the fp64 oracle lives with
the tests (tests/replay_check.py), since product code never runs the oracle.

File format (.npz): q, kv, out, dout as bf16 bit patterns (uint16) of shapes
[T,H,576], [T,1,576], [T,H,512], [T,H,512]; indices int32 [T,1,topk]; lse
float32 [T,H]; scale float64 scalar; cu_seqlens int32 [B+1] (optional).
"""
from __future__ import annotations

import numpy as np
import torch

from bwd_sparse_mla_gb300 import capi

_BF16 = ("q", "kv", "out", "dout")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dump_bwd_call(path, q, kv, out, dout, lse, indices, scale, cu_seqlens=None) -> None:
    """Save the inputs of one backward call (torch tensors, any device)."""
    arrays = {name: _bits(t) for name, t in zip(_BF16, (q, kv, out, dout))}
    arrays["lse"] = lse.detach().float().cpu().numpy()
    arrays["indices"] = indices.detach().to(torch.int32).cpu().numpy()
    arrays["scale"] = np.float64(scale)
    if cu_seqlens is not None:
        arrays["cu_seqlens"] = cu_seqlens.detach().to(torch.int32).cpu().numpy()
    np.savez(path, **arrays)


def load_bwd_call(path) -> dict:
    """Read a dump: numpy arrays (bf16 ones as uint16 bits) and the scale."""
    with np.load(path) as z:
        call = {k: z[k] for k in z.files}
    call["scale"] = float(call["scale"])
    return call


def replay_bwd(call: dict, device="cuda:0", dkv_mode: int = capi.SMLA_DKV_ATOMIC):
    """Re-run the library's backward on a loaded dump.  Returns dq (bf16),
    dkv_f32 and a dict of non-finite counts."""
    dev = torch.device(device)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    q, kv, out, dout = (bf(call[k]) for k in _BF16)
    lse = torch.from_numpy(np.ascontiguousarray(call["lse"], dtype=np.float32)).to(dev)
    idx = torch.from_numpy(np.ascontiguousarray(call["indices"], dtype=np.int32)).to(dev)
    cu = call.get("cu_seqlens")
    cu = None if cu is None else torch.from_numpy(np.ascontiguousarray(cu, dtype=np.int32)).to(dev)
    dq, dkv32, _ = capi.sparse_mla_bwd(q, kv, out, dout, lse, idx, cu, call["scale"], dkv_mode=dkv_mode,
                                       want_bf16_dkv=False)
    torch.cuda.synchronize(dev)
    counts = {
        "dq_nonfinite": int((~torch.isfinite(dq.float())).sum()),
        "dkv_nonfinite": int((~torch.isfinite(dkv32)).sum()),
        "dq_elements": dq.numel(),
        "dkv_elements": dkv32.numel(),
    }
    return dq, dkv32, counts
