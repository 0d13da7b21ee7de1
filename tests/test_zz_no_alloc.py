"""The backward entry point that allocates nothing.

Callers that cannot call cudaMalloc (code inside a memory allocator's own
callbacks, services whose device memory is fixed at start-up) use
sparse_mla_bwd_noalloc: it keeps its Delta scratch in a fixed device array
inside the library instead of a caller-provided workspace.  This file is
named so that pytest collects it last; it passes when run alone in a fresh
process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from bwd_sparse_mla_gb300 import capi
from bwd_sparse_mla_gb300 import workloads as W
from tests.gpu_helpers import assert_close, device_inputs, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H", [16, 128])
def test_noalloc_matches_workspace_backward_twice(H, cuda_device):
    w = W.make_custom(700, H, 256, [300, 400], seed=31, empty_rows=3)
    d = device_inputs(w, cuda_device)
    out, lse = capi.sparse_mla_fwd(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale)
    dq_ref, dkv_ref, dkv16_ref = capi.sparse_mla_bwd(d["q"], d["kv"], out, d["dout"], lse, d["indices"],
                                                     d["cu_seqlens"], w.scale)
    torch.cuda.synchronize()
    lib = capi.load()
    P = ctypes.c_void_p
    for call in range(2):   # two calls in a row share the scratch array
        dq = torch.full_like(dq_ref, float("nan"))
        dkv32 = torch.full_like(dkv_ref, float("nan"))
        dkv16 = torch.full_like(dkv16_ref, float("nan"))
        torch.cuda.synchronize()
        before = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info()[0])
        rc = lib.sparse_mla_bwd_noalloc(
            P(d["q"].data_ptr()), P(d["kv"].data_ptr()), P(out.data_ptr()), P(d["dout"].data_ptr()),
            P(lse.data_ptr()), P(d["indices"].data_ptr()), P(d["cu_seqlens"].data_ptr()), w.T, w.H, w.topk,
            w.B, ctypes.c_float(w.scale), P(dq.data_ptr()), P(dkv32.data_ptr()), P(dkv16.data_ptr()),
            P(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, capi.sparse_mla_last_error()
        torch.cuda.synchronize()
        after = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info()[0])
        if call == 1:   # the first call on a device may load the library's kernels there
            # nothing was allocated: torch's allocator and the device's free memory are unchanged
            assert after == before, f"device memory changed across the call: {before} -> {after}"
        # dq is written by the same kernel with the same inputs: identical
        assert torch.equal(dq, dq_ref)
        # dkv is an fp32 atomic accumulation: equal up to summation order
        assert_close("dkv(noalloc)", to_f64(dkv32), to_f64(dkv_ref), rel_tol=1e-5, abs_tol=1e-4)
        assert torch.equal(dkv16, dkv32.to(torch.bfloat16))


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_device):
    lib = capi.load()
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: the size check comes first
    T = capi.NOALLOC_MAX_ROWS // 128 + 1
    rc = lib.sparse_mla_bwd_noalloc(fake, fake, fake, fake, fake, fake, None, T, 128, 2048, 1, ctypes.c_float(0.04),
                                    fake, fake, None, None)
    assert rc == -22
    assert "no-allocation scratch limit" in capi.sparse_mla_last_error()
