"""Degenerate sizes through the C ABI against the oracle: a single token, a
few tokens, top-k at its minimum (64), every row padding (every block of every
token skipped), and every head count on tiny inputs (the tensor-core kernels
run H < 128 as a 128-row tile with zero rows)."""
import numpy as np
import pytest
import torch

import oracle.sparse_mla_ref as orc
from bwd_sparse_mla_gb300 import capi
from bwd_sparse_mla_gb300 import workloads as W
from tests.gpu_helpers import (LSE_EMPTY_F32, assert_close, device_inputs, f64_to_bf16_dev, oracle_inputs,
                               to_f64)

pytestmark = pytest.mark.gpu


def _run_both(w, dev):
    d = device_inputs(w, dev)
    q, kv, dout = oracle_inputs(w)
    out_ref, lse_ref = orc.sparse_mla_fwd(q, kv, w.indices, w.scale)
    out, lse = capi.sparse_mla_fwd(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale)
    out_in = f64_to_bf16_dev(out_ref, dev)
    lse_in = torch.tensor(lse_ref, dtype=torch.float32, device=dev)
    dq, dkv32, _ = capi.sparse_mla_bwd(d["q"], d["kv"], out_in, d["dout"], lse_in, d["indices"], d["cu_seqlens"],
                                       w.scale)
    torch.cuda.synchronize()
    dq_ref, dkv_ref = orc.sparse_mla_bwd(q, kv, to_f64(out_in), dout, to_f64(lse_in), w.indices, w.scale)
    return (out, lse, dq, dkv32), (out_ref, lse_ref, dq_ref, dkv_ref)


@pytest.mark.parametrize("H", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("T", [1, 3, 70])
def test_tiny_sizes_every_head_count(T, H, cuda_device):
    w = W.make_custom(T, H, 64, [T], seed=71 + T + H)
    (out, lse, dq, dkv), (out_ref, lse_ref, dq_ref, dkv_ref) = _run_both(w, cuda_device)
    assert_close("out", to_f64(out), out_ref, kind="bf16")
    assert_close("lse", to_f64(lse), lse_ref)
    assert_close("dq", to_f64(dq), dq_ref, kind="bf16")
    assert_close("dkv", to_f64(dkv).reshape(T, -1), dkv_ref)


@pytest.mark.parametrize("H", [16, 128])
def test_every_row_padding(H, cuda_device):
    w = W.make_custom(200, H, 128, [200], seed=81)
    w.indices = np.full_like(w.indices, -1)
    (out, lse, dq, dkv), _ = _run_both(w, cuda_device)
    assert int(torch.count_nonzero(out)) == 0
    assert torch.all(lse == LSE_EMPTY_F32)
    assert int(torch.count_nonzero(dq)) == 0
    assert int(torch.count_nonzero(dkv)) == 0


def test_one_valid_slot_per_row(cuda_device):
    """Closed form: with a single valid slot, out = that row's V and dq = 0."""
    w = W.make_custom(150, 128, 64, [150], seed=82)
    idx = np.full_like(w.indices, -1)
    rng = np.random.default_rng(83)
    for t in range(w.T):
        idx[t, 0, rng.integers(0, 64)] = rng.integers(0, t + 1)      # one slot somewhere in the row
    w.indices = idx
    (out, lse, dq, dkv), (out_ref, lse_ref, dq_ref, dkv_ref) = _run_both(w, cuda_device)
    assert_close("out", to_f64(out), out_ref, kind="bf16")
    assert_close("lse", to_f64(lse), lse_ref)
    assert float(dq.abs().max()) < 1e-2          # dS = P (dP - Delta) vanishes with one slot
    assert_close("dkv", to_f64(dkv).reshape(w.T, -1), dkv_ref)
