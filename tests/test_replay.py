"""Single-call dump and replay of a backward call (the slime issue #2201
debugging workflow): the dump round-trips exactly, a replay reproduces the
direct call, and a call whose unnamed kv rows hold NaN/Inf (the kind of
memory a -1 index used to read) replays with no non-finite output and matches
the oracle on every row."""
import numpy as np
import pytest
import torch

import oracle.sparse_mla_ref as orc
from bwd_sparse_mla_gb300 import workloads as W
from tests.gpu_helpers import MAX_ABS, device_inputs, f64_to_bf16_dev, oracle_inputs


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def test_dump_roundtrip_exact(tmp_path):
    from bwd_sparse_mla_gb300 import replay
    w = W.make_custom(64, 8, 64, [64], seed=51, empty_rows=2)
    out = _bf16(w.dout[:, :, :512].copy())      # any bf16 tensor of the right shape
    lse = torch.randn(w.T, w.H)
    path = tmp_path / "call.npz"
    replay.dump_bwd_call(path, _bf16(w.q), _bf16(w.kv), out, _bf16(w.dout), lse,
                         torch.from_numpy(w.indices), w.scale, torch.from_numpy(w.cu_seqlens))
    call = replay.load_bwd_call(path)
    assert np.array_equal(call["q"], w.q) and np.array_equal(call["kv"], w.kv)
    assert np.array_equal(call["dout"], w.dout) and np.array_equal(call["indices"], w.indices)
    assert np.array_equal(call["lse"], lse.numpy()) and call["scale"] == w.scale
    assert np.array_equal(call["cu_seqlens"], w.cu_seqlens)


@pytest.mark.gpu
@pytest.mark.parametrize("H", [16, 128])
def test_replay_matches_direct_call_and_oracle(H, tmp_path, cuda_device):
    from bwd_sparse_mla_gb300 import capi, replay
    from tests import replay_check
    w = W.make_custom(400, H, 256, [150, 250], seed=52, empty_rows=3)
    idx = w.indices.reshape(w.T, -1).copy()
    unnamed = np.array([0, 37, 151, w.T - 1])   # rows no slot names, poisoned below
    idx[np.isin(idx, unnamed)] = -1
    w.indices = idx.reshape(w.T, 1, -1)
    d = device_inputs(w, cuda_device)
    kv_bad = d["kv"].clone()
    ut = torch.from_numpy(unnamed).to(cuda_device)
    kv_bad[ut, 0, 0::2] = float("nan")
    kv_bad[ut, 0, 1::2] = float("inf")
    # the call's out / lse: the oracle forward's (rounded to bf16 / fp32), so that no oracle
    # input comes from the library
    q64, kv64, _ = oracle_inputs(w)
    out_ref, lse_ref = orc.sparse_mla_fwd(q64, kv64, w.indices, w.scale)
    out = f64_to_bf16_dev(out_ref, cuda_device)
    lse = torch.tensor(lse_ref, dtype=torch.float32, device=cuda_device)
    dq, dkv32, _ = capi.sparse_mla_bwd(d["q"], kv_bad, out, d["dout"], lse, d["indices"], d["cu_seqlens"], w.scale)
    torch.cuda.synchronize()
    path = tmp_path / "bad_call.npz"
    replay.dump_bwd_call(path, d["q"], kv_bad, out, d["dout"], lse, d["indices"], w.scale, d["cu_seqlens"])
    dq_r, dkv_r, counts = replay.replay_bwd(replay.load_bwd_call(path), device=cuda_device)
    assert counts["dq_nonfinite"] == 0 and counts["dkv_nonfinite"] == 0
    assert torch.equal(dq_r, dq)                                     # same kernel, same inputs
    assert torch.allclose(dkv_r, dkv32, rtol=1e-5, atol=1e-4)       # fp32 atomics: order may differ
    rep = replay_check.check(path, rows=w.T)
    assert rep["dq_nonfinite"] == 0 and rep["dkv_nonfinite"] == 0
    assert rep["dq_rows_checked"] == w.T
    # the oracle comparison on the finite overlap, with the stated bounds: dq is a bf16
    # output (its values here stay below magnitude 8, so the bound is 2e-2), dkv fp32
    assert rep["dq_max_abs_ref"] < 8.0
    assert rep["dq_max_abs_diff_finite"] <= MAX_ABS and rep["dkv_max_abs_diff_finite"] <= MAX_ABS
