"""GPU checks of the exact invariants the pages state for this path (miles
PR #2079 summary, implementation breakdown items 1-4): padding slots
contribute exactly zero whatever the memory they would address holds, all-
padding rows give exactly-zero output and gradient and a finite LSE, the
clamped padding write to dKV adds nothing, no write lands outside the output
buffers, and finite inputs never give non-finite outputs -- plus a repeated-
run stress test in the spirit of the 50-iteration check on miles PR #1642."""
import numpy as np
import pytest
import torch

import oracle.sparse_mla_ref as orc
from bwd_sparse_mla_gb300 import capi
from bwd_sparse_mla_gb300 import workloads as W
from tests.gpu_helpers import LSE_EMPTY_F32, assert_close, device_inputs, empty_rows, to_f64

pytestmark = pytest.mark.gpu


def _run(d, scale, kv=None, indices=None):
    kv = d["kv"] if kv is None else kv
    indices = d["indices"] if indices is None else indices
    out, lse = capi.sparse_mla_fwd(d["q"], kv, indices, d["cu_seqlens"], scale)
    dq, dkv32, dkv = capi.sparse_mla_bwd(d["q"], kv, out, d["dout"], lse, indices, d["cu_seqlens"], scale)
    torch.cuda.synchronize()
    return out, lse, dq, dkv32, dkv


@pytest.fixture(scope="module", params=[16, 128], ids=["H16", "H128"])
def case(request, cuda_device):
    w = W.make_custom(600, request.param, 128, [250, 350], seed=21, empty_rows=6)
    idx = w.indices.reshape(w.T, -1).copy()
    # rows 0 (the clamp target of -1), 37 and the last row are never named
    poison = np.array([0, 37, w.T - 1])
    idx[np.isin(idx, poison)] = -1
    w.indices = idx.reshape(w.T, 1, -1)
    return w, device_inputs(w, cuda_device), poison


def test_poisoned_unnamed_rows_change_nothing(case):
    w, d, poison = case
    ref = _run(d, w.scale)
    kv_bad = d["kv"].clone()
    pt = torch.from_numpy(poison).to(kv_bad.device)
    kv_bad[pt, 0, ::3] = float("nan")
    kv_bad[pt, 0, 1::3] = float("inf")
    kv_bad[pt, 0, 2::3] = -float("inf")
    got = _run(d, w.scale, kv=kv_bad)
    for name, a, b in zip(("out", "lse", "dq"), ref[:3], got[:3]):
        assert torch.equal(a, b), name
    assert torch.isfinite(got[3]).all()
    assert_close("dkv", to_f64(got[3]), to_f64(ref[3]), rel_tol=1e-5, abs_tol=1e-4)
    assert int(torch.count_nonzero(got[3][pt])) == 0


def test_out_of_range_indices_act_as_padding(case):
    w, d, _ = case
    ref = _run(d, w.scale)
    idx = d["indices"].clone()
    pad = idx == -1
    junk = torch.tensor([-7, w.T, w.T + 100, 2**31 - 1, -2**31], dtype=torch.int32, device=idx.device)
    choice = torch.randint(0, junk.numel(), idx.shape, generator=torch.Generator().manual_seed(3)).to(idx.device)
    idx = torch.where(pad, junk[choice], idx)
    got = _run(d, w.scale, indices=idx)
    for name, a, b in zip(("out", "lse", "dq"), ref[:3], got[:3]):
        assert torch.equal(a, b), name
    assert_close("dkv", to_f64(got[3]), to_f64(ref[3]), rel_tol=1e-5, abs_tol=1e-4)


def test_empty_rows_exact(case):
    w, d, _ = case
    out, lse, dq, dkv32, _ = _run(d, w.scale)
    er = torch.from_numpy(empty_rows(w)).to(out.device)
    assert er.numel() >= 6
    assert int(torch.count_nonzero(out[er])) == 0
    assert int(torch.count_nonzero(dq[er])) == 0
    assert np.all(lse[er].cpu().numpy() == LSE_EMPTY_F32)


def test_never_indexed_rows_get_zero_dkv(case):
    w, d, _ = case
    _, _, _, dkv32, _ = _run(d, w.scale)
    idx = w.indices.reshape(w.T, -1)
    named = np.zeros(w.T, bool)
    named[np.unique(idx[(idx >= 0) & (idx < w.T)])] = True
    z = torch.from_numpy(np.nonzero(~named)[0]).to(dkv32.device)
    assert z.numel() > 0
    assert int(torch.count_nonzero(dkv32[z])) == 0


def test_permuting_a_row_keeps_out_and_lse(case):
    """Shuffling each row's slots (padding lands anywhere, including whole
    padding blocks ahead of the first valid slot) leaves out and lse within
    tolerance of the oracle, which is itself permutation invariant."""
    w, d, _ = case
    g = torch.Generator().manual_seed(5)
    perm = torch.stack([torch.randperm(w.topk, generator=g) for _ in range(w.T)])
    idx_np = np.take_along_axis(w.indices.reshape(w.T, -1), perm.numpy(), axis=1)
    idx = torch.from_numpy(np.ascontiguousarray(idx_np.reshape(w.T, 1, -1))).to(d["q"].device)
    out2, lse2, *_ = _run(d, w.scale, indices=idx)
    out_ref, lse_ref = orc.sparse_mla_fwd(w.q, w.kv, idx_np, w.scale)
    assert_close("out(perm)", to_f64(out2), out_ref, kind="bf16")
    assert_close("lse(perm)", to_f64(lse2), lse_ref)


def test_guard_bands_untouched(case):
    """Outputs live inside larger buffers whose margins hold a NaN pattern;
    the margins must come back bitwise unchanged (an out-of-bounds write in
    front of dKV was one of the failures the pages describe)."""
    w, d, _ = case
    G = 4096  # elements of margin on each side
    dev = d["q"].device

    def guarded(shape, dtype):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * G,), float("nan"), dtype=dtype, device=dev)
        return buf, buf[G:G + n].view(shape)

    T, H = w.T, w.H
    ob, out = guarded((T, H, 512), torch.bfloat16)
    lb, lse = guarded((T, H), torch.float32)
    qb, dq = guarded((T, H, 576), torch.bfloat16)
    kb, dkv32 = guarded((T, 1, 576), torch.float32)
    cb, dkv = guarded((T, 1, 576), torch.bfloat16)
    capi.sparse_mla_fwd(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale, out=out, lse=lse)
    capi.sparse_mla_bwd(d["q"], d["kv"], out, d["dout"], lse, d["indices"], d["cu_seqlens"], w.scale,
                        dq=dq, dkv_f32=dkv32, dkv=dkv)
    torch.cuda.synchronize()
    for buf in (ob, lb, qb, kb, cb):
        assert torch.isnan(buf[:G].float()).all() and torch.isnan(buf[-G:].float()).all()
    for t in (out, lse, dq, dkv32, dkv):
        assert torch.isfinite(t.float()).all()


def test_stress_repeat_50(case):
    w, d, _ = case
    ref = _run(d, w.scale)
    for _ in range(50):
        got = _run(d, w.scale)
        for name, a, b in zip(("out", "lse", "dq"), ref[:3], got[:3]):
            assert torch.equal(a, b), name
        assert torch.isfinite(got[3]).all()
        assert_close("dkv(repeat)", to_f64(got[3]), to_f64(ref[3]), rel_tol=1e-5, abs_tol=1e-4)


def test_check_indices_matches_oracle(cuda_device):
    w = W.make_workload(1)
    idx = w.indices.reshape(w.T, -1).copy()
    idx[3, 0] = 999        # past T
    idx[10, 5] = -9        # negative, not the sentinel
    idx[200, 1] = 255      # in range; the tiny workload is one sequence, so valid
    cu = np.array([0, 100, 256], dtype=np.int32)   # split into two sequences instead
    want = orc.check_indices(idx, cu)
    assert want > 2
    got = capi.sparse_mla_check_indices(torch.from_numpy(idx).to(cuda_device),
                                        torch.from_numpy(cu).to(cuda_device))
    assert got == want


def test_bad_arguments_raise(cuda_device):
    w = W.make_workload(1)
    d = device_inputs(w, cuda_device)
    with pytest.raises(capi.SparseMLAError, match="topk"):
        capi.sparse_mla_fwd(d["q"], d["kv"], d["indices"][:, :, :40].contiguous(), d["cu_seqlens"], w.scale)
