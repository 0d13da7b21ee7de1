"""Row-range calls: a step split into uneven ranges of query rows
(sparse_mla_fwd_rows, sparse_mla_bwd_rows into one zeroed fp32 dKV, then
sparse_mla_dkv_cast) reproduces the whole-step calls -- out, lse and dq bit for
bit, dkv_f32 up to the order of its fp32 additions -- and matches the fp64
oracle.  Rows outside a range are left untouched."""
import numpy as np
import pytest
import torch

import oracle.sparse_mla_ref as orc
from bwd_sparse_mla_gb300 import capi
from bwd_sparse_mla_gb300 import workloads as W
from tests.gpu_helpers import assert_close, device_inputs, f64_to_bf16_dev, oracle_inputs, to_f64

pytestmark = pytest.mark.gpu

CASES = {
    "ragged-H128": lambda: W.make_custom(520, 128, 320, [8, 200, 312], seed=21, empty_rows=3),
    "ragged-H8": lambda: W.make_custom(700, 8, 128, [300, 400], seed=22, empty_rows=2),
    # top-k above the tensor-core kernels' limit: the CUDA-core kernels
    "bigtopk-H8": lambda: W.make_custom(200, 8, 16448, [200], seed=23, empty_rows=2),
}


def _ranges(T):
    """Disjoint, uneven ranges covering [0, T): a single row at each end."""
    b = [0, 1, 1 + T // 3, T - 1, T]
    return [(b[i], b[i + 1] - b[i]) for i in range(len(b) - 1)]


def _bits(t):
    return t.contiguous().view(torch.int16) if t.dtype == torch.bfloat16 else t.contiguous().view(torch.int32)


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request, cuda_device):
    w = CASES[request.param]()
    return w, device_inputs(w, cuda_device), oracle_inputs(w)


def test_fwd_rows_match_the_whole_call(case):
    w, d, _ = case
    out, lse = capi.sparse_mla_fwd(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale)
    out_r = torch.full_like(out, float("nan"))
    lse_r = torch.full_like(lse, float("nan"))
    for t0, nt in _ranges(w.T):
        capi.sparse_mla_fwd_rows(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale, t0, nt, out_r, lse_r)
    torch.cuda.synchronize()
    assert torch.equal(_bits(out_r), _bits(out))
    assert torch.equal(_bits(lse_r), _bits(lse))


def test_fwd_rows_leave_other_rows_alone(case):
    w, d, _ = case
    out_r = torch.full((w.T, w.H, 512), 7.0, dtype=torch.bfloat16, device=d["q"].device)
    lse_r = torch.full((w.T, w.H), 7.0, dtype=torch.float32, device=d["q"].device)
    t0, nt = w.T // 2, 3
    capi.sparse_mla_fwd_rows(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale, t0, nt, out_r, lse_r)
    torch.cuda.synchronize()
    outside = torch.ones(w.T, dtype=torch.bool)
    outside[t0:t0 + nt] = False
    assert torch.all(out_r[outside] == 7.0) and torch.all(lse_r[outside] == 7.0)
    assert not torch.all(lse_r[t0:t0 + nt] == 7.0)


def test_bwd_rows_match_the_whole_call_and_the_oracle(case):
    """Both calls get the oracle's out (bf16) and lse (fp32)."""
    w, d, (q, kv, dout) = case
    out_ref, lse_ref = orc.sparse_mla_fwd(q, kv, w.indices, w.scale)
    dev = d["q"].device
    out_in = f64_to_bf16_dev(out_ref, dev)
    lse_in = torch.tensor(lse_ref, dtype=torch.float32, device=dev)
    dq, dkv32, dkv16 = capi.sparse_mla_bwd(d["q"], d["kv"], out_in, d["dout"], lse_in, d["indices"],
                                           d["cu_seqlens"], w.scale)
    dq_r = torch.full_like(dq, float("nan"))
    dkv32_r = torch.zeros_like(dkv32)
    ws = torch.empty(capi.sparse_mla_bwd_workspace_bytes(w.T, w.H, w.topk), dtype=torch.uint8, device=dev)
    for t0, nt in reversed(_ranges(w.T)):          # any order of the ranges
        capi.sparse_mla_bwd_rows(d["q"], d["kv"], out_in, d["dout"], lse_in, d["indices"], d["cu_seqlens"],
                                 w.scale, t0, nt, dq_r, dkv32_r, ws)
    dkv16_r = capi.sparse_mla_dkv_cast(dkv32_r, torch.empty_like(dkv16))
    dkv16_full_cast = capi.sparse_mla_dkv_cast(dkv32, torch.empty_like(dkv16))
    torch.cuda.synchronize()
    assert torch.equal(_bits(dq_r), _bits(dq))
    # the same contributions, added in another order
    a, b = dkv32_r.double(), dkv32.double()
    assert float((a - b).norm()) <= 1e-5 * float(b.norm()) + 1e-30
    assert torch.equal(_bits(dkv16_full_cast), _bits(dkv16))       # the cast the whole call applies
    assert torch.equal(dkv16_r, dkv32_r.to(torch.bfloat16))
    dq_ref, dkv_ref = orc.sparse_mla_bwd(q, kv, to_f64(out_in), dout, to_f64(lse_in), w.indices, w.scale)
    assert_close("dq", to_f64(dq_r), dq_ref, kind="bf16")
    assert_close("dkv", to_f64(dkv32_r).reshape(w.T, -1), dkv_ref)
    assert np.isfinite(to_f64(dkv16_r)).all()
