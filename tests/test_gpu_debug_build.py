"""The bounds-checked debug build (-DSMLA_DEBUG): every 16-byte gather source and
every scatter destination is checked against its buffer; a failed check records
status 2 and skips the access, it never traps.

The debug library is built into its own folder and run in a child process (this
process has the product library loaded).  Its self-test must report status 2;
on real inputs no check may fire, and the results must equal the product
library's: out, lse and dq bit for bit, dkv bit for bit in the deterministic mode
and within a few fp32 rounding steps in the atomic mode (free reduction order).
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from bwd_sparse_mla_gb300 import build as B
from bwd_sparse_mla_gb300 import capi
from bwd_sparse_mla_gb300 import workloads as W
from tests.gpu_helpers import device_inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# H = 128 and H = 32 (128-row head tile), H = 8 (slots as rows), topk above the
# tensor-core limit (CUDA-core kernels); padding rows in each
CASES = {
    "h128": lambda: W.make_custom(520, 128, 2048, [300, 220], seed=31, empty_rows=3),
    "h32": lambda: W.make_custom(400, 32, 192, [1, 130, 269], seed=32, empty_rows=2),
    "h8": lambda: W.make_custom(700, 8, 256, [350, 350], seed=33, empty_rows=4),
    "bigtopk-h16": lambda: W.make_custom(300, 16, 16448, [300], seed=34, empty_rows=1),
}
MODES = {"atomic": capi.SMLA_DKV_ATOMIC, "det": capi.SMLA_DKV_DETERMINISTIC}

CHILD = r"""
import os, sys
import numpy as np, torch
sys.path.insert(0, {root!r})
from bwd_sparse_mla_gb300 import build as B, capi
from bwd_sparse_mla_gb300 import workloads as W
from tests.gpu_helpers import device_inputs
from tests.test_gpu_debug_build import CASES, MODES, run_case
capi.LIB_PATH = B.debug_paths()[0]
capi.load()
dev = torch.device("cuda:0")
capi.sparse_mla_device_status(clear=True)
capi.sparse_mla_bounds_selftest()
print("selftest", capi.sparse_mla_device_status(clear=True), flush=True)
res = {{}}
for name, make in CASES.items():
    for mode in MODES:
        res.update(run_case(name, make(), mode, dev))
        print(name, mode, "status", capi.sparse_mla_device_status(clear=True), flush=True)
np.savez({out!r}, **res)
"""


def run_case(name, w, mode, dev):
    """Forward and backward of one case through the loaded library; results by key."""
    d = device_inputs(w, dev)
    out, lse = capi.sparse_mla_fwd(d["q"], d["kv"], d["indices"], d["cu_seqlens"], w.scale)
    dq, dkv32, _ = capi.sparse_mla_bwd(d["q"], d["kv"], out, d["dout"], lse, d["indices"], d["cu_seqlens"], w.scale,
                                       dkv_mode=MODES[mode], want_bf16_dkv=False)
    torch.cuda.synchronize()
    k = f"{name}/{mode}/"
    return {k + "out": out.view(torch.int16).cpu().numpy(), k + "lse": lse.cpu().numpy(),
            k + "dq": dq.view(torch.int16).cpu().numpy(), k + "dkv": dkv32.cpu().numpy()}


def test_debug_build_checks_and_matches_the_product_library(tmp_path, cuda_device):
    lib, obj = B.debug_paths()
    B.build(["-DSMLA_DEBUG"], lib=lib, obj=obj)
    out_npz = str(tmp_path / "debug.npz")
    script = CHILD.format(root=ROOT, out=out_npz)
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = dict((ln.rsplit(" ", 1)[0], ln.rsplit(" ", 1)[1]) for ln in r.stdout.strip().splitlines())
    assert lines["selftest"] == "2", r.stdout           # both probes fell outside and were skipped
    for name in CASES:
        for mode in MODES:
            assert lines[f"{name} {mode} status"] == "0", r.stdout   # no check fired on real inputs
    dbg = np.load(out_npz)
    # the product library, in this process, on the same inputs
    with pytest.raises(capi.SparseMLAError):
        capi.sparse_mla_bounds_selftest()               # the product build has no checks to test
    for name, make in CASES.items():
        for mode in MODES:
            ref = run_case(name, make(), mode, cuda_device)
            for key, v in ref.items():
                if key.endswith("dkv") and mode == "atomic":
                    scale = max(1.0, float(np.abs(v).max()))
                    np.testing.assert_allclose(dbg[key], v, rtol=0, atol=1e-5 * scale, err_msg=key)
                else:
                    np.testing.assert_array_equal(dbg[key], v, err_msg=key)
    assert capi.sparse_mla_device_status(clear=True) == 0
