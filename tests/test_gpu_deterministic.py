"""The deterministic dKV mode (an index-sorted segmented reduction).

dkv_f32[r] is the fp32 sum of row r's per-slot contributions taken left to
right in ascending slot order.  Checked here: the same bits on repeated runs and
for any chunking of the query tokens (a workspace that fits only a few tokens'
contributions), dq identical to the atomic mode's, and parity with the oracle
on the same inputs as the atomic mode.  Cases cover the tensor-core path
(H = 16, 64 and 128, with padding holes) and the CUDA-core path (top-k above
the tensor-core limit) with two head groups whose contributions are added in
order (H = 64).
"""
import numpy as np
import pytest
import torch

import oracle.sparse_mla_ref as orc
from bwd_sparse_mla_gb300 import capi
from bwd_sparse_mla_gb300 import workloads as W
from tests.gpu_helpers import assert_close, device_inputs, f64_to_bf16_dev, oracle_inputs, to_f64
from tests.test_gpu_parity import _with_padding_holes

pytestmark = pytest.mark.gpu

CASES = {
    "H16-clustered": lambda: W.make_custom(900, 16, 576, [450, 450], seed=41, kind="clustered", empty_rows=3),
    "H64": lambda: W.make_custom(640, 64, 256, [320, 320], seed=42, empty_rows=2),
    "H128": lambda: W.make_custom(520, 128, 320, [8, 200, 312], seed=43, empty_rows=3),
    "H128-holes": lambda: _with_padding_holes(W.make_custom(500, 128, 512, [500], seed=44, empty_rows=2), 44),
    # top-k above the tensor-core limit: CUDA-core kernels, two head groups added in order
    "H64-bigtopk": lambda: W.make_custom(150, 64, 16448, [150], seed=45, empty_rows=2),
}


def _contribution_bytes_per_token(w):
    # the tensor-core kernels store one contribution per slot; above their top-k limit the
    # CUDA-core kernels store one per head group of 32 heads (one for H <= 16)
    groups = 1 if (w.topk <= 16384 or w.H <= 16) else w.H // 32
    return groups * w.topk * 576 * 4


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request, cuda_device):
    w = CASES[request.param]()
    d = device_inputs(w, cuda_device)
    q, kv, dout = oracle_inputs(w)
    out_ref, lse_ref = orc.sparse_mla_fwd(q, kv, w.indices, w.scale)
    # both sides get the oracle's out rounded to bf16 and its lse rounded to fp32
    out_in = f64_to_bf16_dev(out_ref, cuda_device)
    lse_in = torch.tensor(lse_ref, dtype=torch.float32, device=cuda_device)
    dq_ref, dkv_ref = orc.sparse_mla_bwd(q, kv, to_f64(out_in), dout, to_f64(lse_in), w.indices, w.scale)
    return w, d, out_in, lse_in, dq_ref, dkv_ref


def _bwd(w, d, out_in, lse_in, mode, workspace=None):
    dq, dkv32, dkv16 = capi.sparse_mla_bwd(d["q"], d["kv"], out_in, d["dout"], lse_in, d["indices"],
                                           d["cu_seqlens"], w.scale, dkv_mode=mode, workspace=workspace)
    torch.cuda.synchronize()
    return dq, dkv32, dkv16


def test_deterministic_bits_repeat_and_match_oracle(case):
    w, d, out_in, lse_in, dq_ref, dkv_ref = case
    dq1, dkv1, dkv16 = _bwd(w, d, out_in, lse_in, capi.SMLA_DKV_DETERMINISTIC)
    for _ in range(3):
        dq2, dkv2, _ = _bwd(w, d, out_in, lse_in, capi.SMLA_DKV_DETERMINISTIC)
        assert torch.equal(dkv1, dkv2)
        assert torch.equal(dq1, dq2)
    assert torch.equal(dkv16, dkv1.to(torch.bfloat16))
    assert_close("dq", to_f64(dq1), dq_ref, kind="bf16")
    assert_close("dkv", to_f64(dkv1).reshape(w.T, -1), dkv_ref)
    # rows no valid slot names stay exactly 0
    idx = w.indices.reshape(w.T, -1)
    named = np.zeros(w.T, bool)
    named[np.unique(idx[(idx >= 0) & (idx < w.T)])] = True
    assert np.all(to_f64(dkv1).reshape(w.T, -1)[~named] == 0.0)


def test_deterministic_against_atomic(case):
    w, d, out_in, lse_in, _, _ = case
    dq_a, dkv_a, _ = _bwd(w, d, out_in, lse_in, capi.SMLA_DKV_ATOMIC)
    dq_d, dkv_d, _ = _bwd(w, d, out_in, lse_in, capi.SMLA_DKV_DETERMINISTIC)
    assert torch.equal(dq_a, dq_d)              # dq does not depend on the dKV mode
    # the same fp32 sums in another order
    assert_close("dkv(det vs atomic)", to_f64(dkv_d), to_f64(dkv_a), rel_tol=1e-5, abs_tol=1e-4)


@pytest.mark.parametrize("chunk_tokens", [1, 7])
def test_deterministic_bits_do_not_depend_on_chunking(case, chunk_tokens):
    w, d, out_in, lse_in, _, _ = case
    _, dkv_full, _ = _bwd(w, d, out_in, lse_in, capi.SMLA_DKV_DETERMINISTIC)
    full = capi.sparse_mla_bwd_workspace_bytes(w.T, w.H, w.topk, capi.SMLA_DKV_DETERMINISTIC)
    per_tok = _contribution_bytes_per_token(w)
    default_tokens = min(w.T, max(1, (4 << 30) // per_tok))   # the library's default chunk (4 GiB)
    fixed = full - default_tokens * per_tok
    ws = torch.empty(fixed + chunk_tokens * per_tok, dtype=torch.uint8, device=d["q"].device)
    _, dkv_small, _ = _bwd(w, d, out_in, lse_in, capi.SMLA_DKV_DETERMINISTIC, workspace=ws)
    assert torch.equal(dkv_small, dkv_full)
