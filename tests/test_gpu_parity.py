"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small workloads are compared element by element on every output; the five
full-size workloads are compared on a stratified row sample (out, lse, dq),
and dkv is compared in full with dO zeroed outside the sampled rows, so the
oracle can compute the exact dkv from the sampled rows alone.
"""
import numpy as np
import pytest
import torch

import oracle.sparse_mla_ref as orc
from bwd_sparse_mla_gb300 import capi
from bwd_sparse_mla_gb300 import workloads as W
from tests.gpu_helpers import (LSE_EMPTY_F32, assert_close, device_inputs, empty_rows,
                               f64_to_bf16_dev, oracle_inputs, to_f64)

pytestmark = pytest.mark.gpu

def _with_padding_holes(w, seed):
    """Moves each row's valid slots to random positions outside 64-slot blocks 1, 4 and 6, so
    that whole blocks of padding sit between valid ones (the kernels skip such blocks)."""
    rng = np.random.default_rng(seed)
    idx = w.indices.reshape(w.T, w.topk)
    out = np.full_like(idx, -1)
    allowed = np.array([c for c in range(w.topk) if c // 64 not in (1, 4, 6)])
    for r in range(w.T):
        v = idx[r][idx[r] >= 0]
        v = v[: allowed.size]
        out[r, np.sort(rng.choice(allowed, v.size, replace=False))] = v
    w.indices = out.reshape(w.T, 1, w.topk)
    return w


def _with_empty_run(w, lo, hi):
    """Rows lo..hi-1 get only padding: every persistent CTA (pair) then meets a run of
    consecutive all-padding tokens between tokens with valid slots."""
    idx = w.indices.reshape(w.T, w.topk)
    idx[lo:hi] = -1
    w.indices = idx.reshape(w.T, 1, w.topk)
    return w


SMALL = {
    "cfg1-tiny": lambda: W.make_workload(1),
    "ragged-H8": lambda: W.make_custom(1000, 8, 128, [300, 576, 124], seed=11, empty_rows=5),
    "ragged-H16-clustered": lambda: W.make_custom(1200, 16, 576, [600, 600], seed=12, kind="clustered",
                                                  empty_rows=3),
    "ragged-H32": lambda: W.make_custom(700, 32, 192, [1, 130, 569], seed=13, empty_rows=4),
    "ragged-H64": lambda: W.make_custom(640, 64, 256, [320, 320], seed=14, empty_rows=2),
    "ragged-H128-bigq": lambda: W.make_custom(520, 128, 320, [8, 200, 312], seed=15, empty_rows=3,
                                              q_std=8.0),
    # whole blocks of padding between valid slots
    "holes-H128": lambda: _with_padding_holes(W.make_custom(600, 128, 512, [600], seed=16, empty_rows=2), 16),
    # top-k above the tensor-core kernels' limit (runs the CUDA-core kernels)
    "bigtopk-H128": lambda: W.make_custom(260, 128, 16448, [260], seed=17, empty_rows=2),
    "bigtopk-H8": lambda: W.make_custom(200, 8, 16448, [200], seed=18, empty_rows=2),
    # runs of all-padding tokens in every CTA's token list, between tokens with valid slots
    "empty-run-H128": lambda: _with_empty_run(W.make_custom(1200, 128, 256, [1200], seed=19), 300, 900),
    "empty-run-H64": lambda: _with_empty_run(W.make_custom(1200, 64, 320, [700, 500], seed=20), 250, 950),
    "empty-run-H8": lambda: _with_empty_run(W.make_custom(1400, 8, 256, [1400], seed=21), 300, 1100),
}


@pytest.fixture(scope="module", params=sorted(SMALL))
def small(request, cuda_device):
    w = SMALL[request.param]()
    d = device_inputs(w, cuda_device)
    q, kv, dout = oracle_inputs(w)
    out_ref, lse_ref = orc.sparse_mla_fwd(q, kv, w.indices, w.scale)
    return w, d, (q, kv, dout), (out_ref, lse_ref)


def test_fwd_small(small):
    w, d, _, (out_ref, lse_ref) = small
    out, lse = capi.sparse_mla_fwd(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale)
    torch.cuda.synchronize()
    out_g, lse_g = to_f64(out), to_f64(lse)
    assert_close("out", out_g, out_ref, kind="bf16")
    assert_close("lse", lse_g, lse_ref)
    er = empty_rows(w)
    assert er.size > 0
    assert np.all(out_g[er] == 0.0)
    assert np.all(lse.cpu().numpy()[er] == LSE_EMPTY_F32)


def test_bwd_small(small):
    """Backward alone: both sides get the oracle's out (bf16) and lse (fp32)."""
    w, d, (q, kv, dout), (out_ref, lse_ref) = small
    out_in = f64_to_bf16_dev(out_ref, d["q"].device)
    lse_in = torch.tensor(lse_ref, dtype=torch.float32, device=d["q"].device)
    dq, dkv32, dkv16 = capi.sparse_mla_bwd(d["q"], d["kv"], out_in, d["dout"], lse_in, d["indices"],
                                           d["cu_seqlens"], w.scale)
    torch.cuda.synchronize()
    dq_ref, dkv_ref = orc.sparse_mla_bwd(q, kv, to_f64(out_in), dout, to_f64(lse_in), w.indices, w.scale)
    assert_close("dq", to_f64(dq), dq_ref, kind="bf16")
    assert_close("dkv", to_f64(dkv32).reshape(w.T, -1), dkv_ref)
    # the bf16 copy is the round-to-nearest-even cast of the fp32 accumulator
    assert torch.equal(dkv16, dkv32.to(torch.bfloat16))
    er = empty_rows(w)
    assert np.all(to_f64(dq)[er] == 0.0)
    idx = w.indices.reshape(w.T, -1)
    named = np.zeros(w.T, bool)
    named[np.unique(idx[(idx >= 0) & (idx < w.T)])] = True
    assert np.all(to_f64(dkv32).reshape(w.T, -1)[~named] == 0.0)


def test_fwd_bwd_chain_small(small):
    """GPU forward feeding GPU backward, at every head count and logit scale.

    The forward's out / lse are compared with the oracle forward.  The backward
    takes out and lse as given inputs (the kernel call in slime issue #2201,
    "Strongest repro evidence", passes tl_out and tl_lse), so its results are
    compared with the oracle backward given the same bf16 out and fp32 lse."""
    w, d, (q, kv, dout), (out_ref, lse_ref) = small
    out, lse = capi.sparse_mla_fwd(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale)
    dq, dkv32, _ = capi.sparse_mla_bwd(d["q"], d["kv"], out, d["dout"], lse, d["indices"],
                                       d["cu_seqlens"], w.scale)
    torch.cuda.synchronize()
    assert_close("out(chain)", to_f64(out), out_ref, kind="bf16")
    assert_close("lse(chain)", to_f64(lse), lse_ref)
    dq_ref, dkv_ref = orc.sparse_mla_bwd(q, kv, to_f64(out), dout, to_f64(lse), w.indices, w.scale)
    assert_close("dq(chain)", to_f64(dq), dq_ref, kind="bf16")
    assert_close("dkv(chain)", to_f64(dkv32).reshape(w.T, -1), dkv_ref)


FULL_SAMPLE = {2: 512, 3: 512, 4: 384, 5: 256}


@pytest.mark.parametrize("cfg,dkv_mode", [(2, 0), (3, 0), (3, 1), (4, 0), (5, 0), (5, 1)],
                         ids=["cfg2", "cfg3", "cfg3-deterministic", "cfg4", "cfg5", "cfg5-deterministic"])
def test_full_size_sampled(cfg, dkv_mode, cuda_device):
    w = W.make_workload(cfg)
    rows = W.sample_rows(w, FULL_SAMPLE[cfg])
    d = device_inputs(w, cuda_device)
    out, lse = capi.sparse_mla_fwd(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    out_ref, lse_ref = orc.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, rows=rows)
    rt = torch.from_numpy(rows).to(cuda_device)
    assert_close("out", to_f64(out[rt]), out_ref, kind="bf16")
    assert_close("lse", to_f64(lse[rt]), lse_ref)
    er = empty_rows(w)
    assert np.all(to_f64(out[torch.from_numpy(er).to(cuda_device)]) == 0.0)
    assert np.all(lse[torch.from_numpy(er).to(cuda_device)].cpu().numpy() == LSE_EMPTY_F32)

    # backward with dO zeroed outside the sample; sampled rows get the oracle's out/lse
    out_in = out.clone()
    out_in[rt] = f64_to_bf16_dev(out_ref, cuda_device)
    lse_in = lse.clone()
    lse_in[rt] = torch.tensor(lse_ref, dtype=torch.float32, device=cuda_device)
    del out, lse
    dout_m = torch.zeros_like(d["dout"])
    dout_m[rt] = d["dout"][rt]
    dq, dkv32, _ = capi.sparse_mla_bwd(d["q"], d["kv"], out_in, dout_m, lse_in, d["indices"],
                                       d["cu_seqlens"], w.scale, dkv_mode=dkv_mode, want_bf16_dkv=False)
    torch.cuda.synchronize()
    dq_ref, dkv_ref = orc.sparse_mla_bwd(w.q, w.kv, to_f64(out_in[rt]), w.dout, to_f64(lse_in[rt]),
                                         w.indices, w.scale, rows=rows)
    assert_close("dq", to_f64(dq[rt]), dq_ref, kind="bf16")
    # rows outside the sample have dO = 0, hence dS = 0 and dq exactly 0
    nz = torch.cat([torch.count_nonzero(dq[i:i + 4096], dim=(1, 2)) for i in range(0, w.T, 4096)])
    nz[rt] = 0
    assert int(nz.sum()) == 0
    assert_close("dkv", to_f64(dkv32).reshape(w.T, -1), dkv_ref)
