"""Replay a dumped backward call and check it against the fp64 oracle.

    python -m tests.replay_check call.npz [--rows N] [--full]

Reports, as the slime issue #2201 workflow does for a bad call: the number of
non-finite entries of dq and dkv from the library, and the largest difference
from the oracle on the finite overlap -- dq on a sample of rows (every row with
--full), dkv in full when the dump is small enough or with --full.
"""
from __future__ import annotations

import argparse
import json

import numpy as np

import oracle.sparse_mla_ref as orc
from bwd_sparse_mla_gb300 import replay


def check(path, rows: int = 256, full: bool = False, seed: int = 0, device="cuda:0") -> dict:
    call = replay.load_bwd_call(path)
    dq, dkv32, counts = replay.replay_bwd(call, device=device)
    T = call["q"].shape[0]
    if full or T <= rows:
        sample = np.arange(T)
    else:
        sample = np.sort(np.random.default_rng(seed).choice(T, size=rows, replace=False))
    q, kv, out, dout = call["q"], call["kv"], call["out"], call["dout"]
    dq_ref, dkv_ref = orc.sparse_mla_bwd(q, kv, out[sample], dout, call["lse"][sample].astype(np.float64),
                                         call["indices"], call["scale"], rows=sample)
    dq_g = dq.float().cpu().numpy().astype(np.float64)[sample]
    fin = np.isfinite(dq_g)
    report = dict(counts)
    report["dq_rows_checked"] = int(sample.size)
    report["dq_max_abs_diff_finite"] = float(np.abs(dq_g - dq_ref)[fin].max()) if fin.any() else 0.0
    report["dq_max_abs_ref"] = float(np.abs(dq_ref).max()) if dq_ref.size else 0.0
    if sample.size == T:       # every row's contribution is in the oracle's dkv
        dkv_g = dkv32.cpu().numpy().astype(np.float64).reshape(T, -1)
        fin = np.isfinite(dkv_g)
        report["dkv_max_abs_diff_finite"] = float(np.abs(dkv_g - dkv_ref)[fin].max()) if fin.any() else 0.0
    return report


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("path")
    ap.add_argument("--rows", type=int, default=256)
    ap.add_argument("--full", action="store_true")
    args = ap.parse_args()
    print(json.dumps(check(args.path, rows=args.rows, full=args.full)))


if __name__ == "__main__":
    main()
