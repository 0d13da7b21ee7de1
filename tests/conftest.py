import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU work (oracle on big samples)")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """After every GPU test: no bounded wait inside a tensor-core kernel gave up."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    from bwd_sparse_mla_gb300 import capi
    assert capi.sparse_mla_device_status(clear=True) == 0, "a kernel wait timed out"


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Per-output errors of every GPU-vs-oracle comparison made in this session."""
    import sys
    mod = sys.modules.get("tests.gpu_helpers")
    recs = getattr(mod, "PARITY_RECORDS", None) if mod else None
    if not recs:
        return
    tr = terminalreporter
    tr.section("parity errors (relative Frobenius, max abs, worst |err|/bound)")
    for r in recs:
        tr.write_line(f"{r['test']:<72.72} {r['output']:<20.20} {r['kind']:<4} rel_fro={r['rel_fro']:.2e} "
                      f"max_abs={r['max_abs']:.2e} ratio={r['bound_ratio']:.3f} max|ref|={r['max_abs_ref']:.3g}")
