"""Failure detection of the tensor-core kernels, tested without a GPU fault.

Every wait inside those kernels is bounded: after its limit it records a
status word and the kernel returns, so a lost peer or a copy that never lands
shows up as a status the host reads, not as a hung GPU.  The self-test entry
point makes one such wait run out (a barrier that nothing releases); the test
reads the status, clears it and checks that the same context still computes
correct results.
"""
import time

import pytest
import torch

from bwd_sparse_mla_gb300 import capi
from bwd_sparse_mla_gb300 import workloads as W
from oracle import sparse_mla_ref as ref
from tests.gpu_helpers import assert_close, device_inputs, to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives(cuda_device):
    assert capi.sparse_mla_device_status(clear=True) == 0
    t0 = time.perf_counter()
    capi.sparse_mla_wait_selftest()
    assert capi.sparse_mla_device_status() == 1          # the wait gave up and said so
    elapsed = time.perf_counter() - t0
    assert 0.9 < elapsed < 30.0, elapsed                 # it waited about its 1 s limit, then returned
    assert capi.sparse_mla_device_status(clear=True) == 1
    assert capi.sparse_mla_device_status() == 0          # cleared

    # the context is still usable: an H=128 forward right after matches the oracle
    w = W.make_custom(300, 128, 256, [300], seed=41, empty_rows=2)
    d = device_inputs(w, cuda_device)
    out, lse = capi.sparse_mla_fwd(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale)
    torch.cuda.synchronize()
    assert capi.sparse_mla_device_status() == 0
    rows = list(range(0, w.T, 7))
    o_ref, lse_ref = ref.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, rows=rows)
    assert_close("out", to_f64(out)[rows], o_ref, kind="bf16")
    assert_close("lse", to_f64(lse)[rows], lse_ref)
