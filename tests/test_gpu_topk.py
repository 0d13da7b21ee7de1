"""Top-k index selection (Megatron-Bridge PR #17: top-k capped at the causal
candidate count, padded with -1) against the oracle, bit-exact: ties, NaN,
ragged sequences, sequences longer than ncols, and the indices feeding the
sparse MLA forward."""
import numpy as np
import pytest
import torch

import oracle.sparse_mla_ref as orc
import oracle.topk_ref as tk
from bwd_sparse_mla_gb300 import capi
from bwd_sparse_mla_gb300 import workloads as W
from tests.gpu_helpers import assert_close, device_inputs, to_f64

pytestmark = pytest.mark.gpu


def _scores(seed, T, ncols, tie_levels=None, nan_frac=0.0):
    rng = np.random.default_rng(seed)
    s = rng.standard_normal((T, ncols)).astype(np.float32)
    if tie_levels:
        s = (np.round(s * tie_levels) / tie_levels).astype(np.float32)   # many exact ties
    s[rng.random((T, ncols)) < nan_frac] = np.nan
    return s


@pytest.mark.parametrize("T,ncols,topk,lens,ties,nan", [
    (700, 600, 128, [300, 400], None, 0.0),
    (700, 600, 128, [300, 400], 4, 0.02),          # ties and NaN
    (900, 256, 64, [1, 2, 400, 497], 8, 0.0),       # sequences longer than ncols are capped
    (4096, 4096, 2048, [4096], None, 0.0),          # headline-like width
    (513, 512, 8192, [513], 2, 0.01),               # topk wider than any candidate list
    (3000, 3000, 4096, [3000], None, 0.0),          # k up to 3000: four sorted pairs a thread
    (6000, 6000, 8192, [1000, 5000], 4, 0.01),      # k up to 5000: eight sorted pairs a thread
    (4096, 4096, 1024, [4096], 1, 0.01),            # ties at the threshold overflow the buffer: ordered collect
    (3000, 3000, 2048, [3000], 1e-9, 0.0),          # every score 0 or -0: all tie, columns in order
])
def test_topk_matches_oracle(T, ncols, topk, lens, ties, nan, cuda_device):
    s = _scores(7 + T + topk, T, ncols, ties, nan)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    got = capi.sparse_mla_topk(torch.from_numpy(s).to(cuda_device), torch.from_numpy(cu).to(cuda_device), topk)
    torch.cuda.synchronize()
    ref = tk.topk_indices(s.astype(np.float64), cu, topk)
    assert np.array_equal(got.cpu().numpy(), ref)


def test_topk_indices_feed_sparse_mla(cuda_device):
    """Indices from the selection drive the forward; the oracle forward on the
    oracle's own indices gives the same out and lse."""
    w = W.make_custom(600, 16, 256, [250, 350], seed=61)
    s = _scores(62, w.T, 400, tie_levels=16)
    idx_ref = tk.topk_indices(s.astype(np.float64), w.cu_seqlens, w.topk)
    d = device_inputs(w, cuda_device)
    idx = capi.sparse_mla_topk(torch.from_numpy(s).to(cuda_device), d["cu_seqlens"], w.topk)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    out, lse = capi.sparse_mla_fwd(d["q"], d["kv"], idx, d["cu_seqlens"], w.scale)
    torch.cuda.synchronize()
    out_ref, lse_ref = orc.sparse_mla_fwd(w.q, w.kv, idx_ref, w.scale)
    assert_close("out", to_f64(out), out_ref, kind="bf16")
    assert_close("lse", to_f64(lse), lse_ref)
    assert capi.sparse_mla_check_indices(idx, d["cu_seqlens"]) == 0     # every index in its own sequence
