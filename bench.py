"""Benchmark of the sparse MLA hot path (forward + backward) on GB300.

One step = sparse_mla_fwd then sparse_mla_bwd (Delta pass, dKV zeroing, main
backward kernel, dKV cast) over the headline workload: T=65536 packed tokens,
H=128, topk=2048, ragged log-uniform sequence lengths in [128, 32768],
q ~ N(0, 8^2), 1% all-padding rows.  Inputs are seeded synthetic data resident
in HBM when the timed region starts; L2 is flushed (a 256 MiB write) before
every timed step, outside the step's CUDA events.

Prints one JSON line.  `--impl reference` times the fp64 CPU oracle instead,
on a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bwd_sparse_mla_gb300 import workloads as W  # noqa: E402

METRIC = "sparse-MLA fwd+bwd tokens/s at H=128, topk=2048 (T=65536)"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GATHER_BYTES_PER_SLOT = 1152          # one 576-wide bf16 KV row per valid slot
FWD_FLOP_PER_SLOT_HEAD = 2 * 1088     # QK^T over 576 + PV over 512
BWD_FLOP_PER_SLOT_HEAD = 2 * 2752     # S 576 + dP 512 + dQ 576 + dKV 512+576
DKV_RED_BYTES_PER_SLOT = 2304         # fp32 scatter of a 576-wide row


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, f"{pre}{k}.")
                else:
                    flat[pre[:-1]] = x
            walk(d)
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                for k, v in flat.items():
                    if k.split(".")[-1] == key and isinstance(v, (int, float)):
                        out[key] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None, log_path: str | None):
        self.proc = None
        self.log_path = log_path
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if bus_id:
            cmd += ["-i", bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        if self.log_path:
            try:
                with open(self.log_path, "w") as f:
                    f.write(self.FIELDS + "\n" + out)
            except Exception:
                pass
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "samples": len(sm),
                "reasons": sorted(reasons)}


def bus_id_of(dev) -> str | None:
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:
        return None


def oracle_tokens_per_s(w, target_s: float, seed: int = 17):
    """Time the fp64 oracle (forward then backward) on a bounded row sample."""
    import oracle.sparse_mla_ref as orc
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(w.T, size=2, replace=False))
    t0 = time.perf_counter()
    o, l = orc.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, rows=rows)
    orc.sparse_mla_bwd(w.q, w.kv, o, w.dout, l, w.indices, w.scale, rows=rows)
    per_row = (time.perf_counter() - t0) / rows.size
    n = int(max(2, min(w.T, target_s / max(per_row, 1e-6))))
    rows = np.sort(rng.choice(w.T, size=n, replace=False))
    t0 = time.perf_counter()
    o, l = orc.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, rows=rows)
    orc.sparse_mla_bwd(w.q, w.kv, o, w.dout, l, w.indices, w.scale, rows=rows)
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        th = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if th:
            return int(max(th))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args):
    """Reference arm: the fp64 CPU oracle, as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = W.make_workload(args.config, values=False)
    rng = np.random.default_rng(99)
    n_rows = args.ref_rows
    samples = [np.sort(rng.choice(w.T, size=n_rows, replace=False)) for _ in range(args.warmup + args.steps)]
    W.draw_values(w, rows=np.concatenate(samples))
    import oracle.sparse_mla_ref as orc
    times = []
    for i, rows in enumerate(samples):
        t0 = time.perf_counter()
        o, l = orc.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, rows=rows)
        orc.sparse_mla_bwd(w.q, w.kv, o, w.dout, l, w.indices, w.scale, rows=rows)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    step_s = float(np.mean(times))
    value = n_rows / step_s
    cores = blas_threads()
    sample = f"{n_rows} random rows of the {w.name} workload per step (fwd+bwd, fp64)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "topk": w.topk, "rows_per_step": n_rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


MODE_NAMES = {0: "atomic", 1: "deterministic (index-sorted segmented reduction)"}


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over the ranks of the default process
    group (the values themselves without one): replicas report the slowest
    rank's times."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def replica_throughput(tokens_per_rank, world, ms):
    """Whole-job tokens/s of `world` replicas that each processed
    tokens_per_rank tokens, the slowest taking `ms` milliseconds."""
    return world * tokens_per_rank / (ms / 1e3)


def run_ours(args):
    import torch
    import torch.distributed as dist
    from bwd_sparse_mla_gb300 import capi

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    capi.load()

    if args.tokens:
        w = W.make_workload(args.config, values=False)
        W.draw_values(w, rows=range(args.tokens))
        w = W.truncate(w, args.tokens)
    else:
        w = W.make_workload(args.config)
    n_valid = w.n_valid()
    T, H, topk = w.T, w.H, w.topk

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    h_q, h_kv, h_dout = bf(w.q), bf(w.kv), bf(w.dout)
    h_idx = torch.from_numpy(np.ascontiguousarray(w.indices))
    h_cu = torch.from_numpy(w.cu_seqlens)
    q, kv, dout = h_q.to(dev), h_kv.to(dev), h_dout.to(dev)
    idx, cu = h_idx.to(dev), h_cu.to(dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    dq = torch.empty((T, H, 576), dtype=torch.bfloat16, device=dev)
    dkv32 = torch.empty((T, 1, 576), dtype=torch.float32, device=dev)
    dkv = torch.empty((T, 1, 576), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(capi.sparse_mla_bwd_workspace_bytes(T, H, topk, args.dkv_mode), 256), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        capi.sparse_mla_fwd(q, kv, idx, cu, w.scale, out=out, lse=lse)
        capi.sparse_mla_bwd(q, kv, out, dout, lse, idx, cu, w.scale, dkv_mode=args.dkv_mode, dq=dq, dkv_f32=dkv32,
                            dkv=dkv, workspace=ws)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(bus_id_of(dev), args.clocks_csv)
    launches0 = capi.sparse_mla_launch_count()
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.zero_()
        ev[k][0].record(stream)
        capi.sparse_mla_fwd(q, kv, idx, cu, w.scale, out=out, lse=lse)
        ev[k][1].record(stream)
        capi.sparse_mla_bwd(q, kv, out, dout, lse, idx, cu, w.scale, dkv_mode=args.dkv_mode, dq=dq, dkv_f32=dkv32,
                            dkv=dkv, workspace=ws)
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    launches = capi.sparse_mla_launch_count() - launches0
    clocks = sampler.stop()
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    bwd_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    ms = fwd_ms + bwd_ms
    ms, fwd_ms, bwd_ms = max_over_ranks([ms, fwd_ms, bwd_ms], dev)
    value = replica_throughput(T, world, ms)

    # finite-output check of the last timed step (outside the timed region)
    finite = bool(torch.isfinite(lse).all()) and bool(torch.isfinite(dkv32).all())

    peaks, peak_src = load_peaks()
    fwd_flop = FWD_FLOP_PER_SLOT_HEAD * H * n_valid
    bwd_flop = BWD_FLOP_PER_SLOT_HEAD * H * n_valid
    gbytes = GATHER_BYTES_PER_SLOT * n_valid
    tflops_peak = peaks["bf16_tflops_sustained"]
    hbm = peaks["hbm_gbs"]

    def bound_ms(flop):
        return max(flop / (tflops_peak * 1e12), gbytes / (hbm * 1e9)) * 1e3

    ridge = tflops_peak * 1e12 / (hbm * 1e9)
    bwd_tensor = bwd_flop / gbytes > ridge
    if bwd_tensor:
        achieved = bwd_flop / (bwd_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tflops_peak, "unit": "TFLOP/s",
                "frac": achieved / tflops_peak}
    else:
        achieved = gbytes / (bwd_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm}
    roof.update({
        "kernel": "sparse_mla_bwd call (Delta + dKV zero + main backward + dKV cast)",
        "peak_source": f"{peak_src} bf16_tflops_sustained / hbm_gbs",
        "algorithmic_per_launch": {"flop": bwd_flop, "gathered_kv_bytes": gbytes},
        "traffic": None,
    })
    tr = traffic_record()
    if tr is not None:
        roof["traffic"] = tr["dram_bytes_per_launch"]
        roof["traffic_note"] = tr["note"]

    # the other dKV mode, timed after the main region with the same L2 flush
    other = None
    if args.other_mode_steps > 0:
        omode = 1 - args.dkv_mode
        ws_o = torch.empty(max(capi.sparse_mla_bwd_workspace_bytes(T, H, topk, omode), 256), dtype=torch.uint8,
                           device=dev)
        capi.sparse_mla_bwd(q, kv, out, dout, lse, idx, cu, w.scale, dkv_mode=omode, dq=dq, dkv_f32=dkv32, dkv=dkv,
                            workspace=ws_o)
        oev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.other_mode_steps)]
        for k in range(args.other_mode_steps):
            flush.zero_()
            oev[k][0].record(stream)
            capi.sparse_mla_bwd(q, kv, out, dout, lse, idx, cu, w.scale, dkv_mode=omode, dq=dq, dkv_f32=dkv32,
                                dkv=dkv, workspace=ws_o)
            oev[k][1].record(stream)
        torch.cuda.synchronize()
        o_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in oev]))
        other = {"dkv_mode": MODE_NAMES[omode], "ms": o_ms, "tflops": bwd_flop / (o_ms * 1e-3) / 1e12,
                 "workspace_bytes": int(ws_o.numel()), "steps": args.other_mode_steps}
        del ws_o

    e2e = None
    if rank == 0 or world > 1:
        e2e = run_e2e(args, capi, w, dev, h_q, h_kv, h_dout, h_idx, h_cu)
        e2e["matches_device_step"] = same_results(e2e.pop("_host"), (out, lse, dq, dkv), dev)
        if world > 1:
            e2e["ms_per_step"] = max_over_ranks([e2e["ms_per_step"]], dev)[0]
            e2e["value"] = replica_throughput(T, world, e2e["ms_per_step"])

    # the other workloads, measured after the headline's timed region (rank 0 only)
    others = None
    if rank == 0 and args.workloads != "none":
        del out, lse, dq, dkv32, dkv, ws, flush, q, kv, dout, idx, cu
        torch.cuda.empty_cache()
        others = {}
        for c in [int(x) for x in args.workloads.split(",") if x]:
            others[str(c)] = time_workload(capi, c, dev, args.workload_steps, 2, peaks)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, n, dt = oracle_tokens_per_s(w, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": f"{n} random rows of the workload, fwd+bwd in fp64 ({dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "T": T, "H": H, "topk": topk, "valid_slots": n_valid,
                       "sequences": w.B, "l2": "flushed before every timed step (256 MiB write)",
                       "parallelism": "replicas" if world > 1 else "single-gpu"},
            "fwd": {"ms": fwd_ms, "tflops": fwd_flop / (fwd_ms * 1e-3) / 1e12,
                    "roofline_frac": bound_ms(fwd_flop) / fwd_ms, "gathered_kv_gbs": gbytes / (fwd_ms * 1e-3) / 1e9},
            "bwd": {"ms": bwd_ms, "tflops": bwd_flop / (bwd_ms * 1e-3) / 1e12,
                    "roofline_frac": bound_ms(bwd_flop) / bwd_ms, "gathered_kv_gbs": gbytes / (bwd_ms * 1e-3) / 1e9,
                    "dkv_mode": MODE_NAMES[args.dkv_mode], "dkv_scatter_bytes": DKV_RED_BYTES_PER_SLOT * n_valid},
            "bwd_other_dkv_mode": other,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks,
            "workloads": others,
            "gpu_launches": launches,
            "wall_s_timed": wall,
            "outputs_finite": finite,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def time_workload(capi, cfg: int, dev, steps: int, warmup: int, peaks: dict):
    """fwd and bwd of workload `cfg` (inputs resident in HBM, L2 flushed before
    each step): times, TFLOP/s, tokens/s, fractions of the roofline and the
    achieved rate of gathered KV bytes.  Run after the headline timed region."""
    import torch
    w = W.make_workload(cfg)
    T, H, topk = w.T, w.H, w.topk
    n_valid = w.n_valid()

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    q, kv, dout = bf(w.q), bf(w.kv), bf(w.dout)
    idx = torch.from_numpy(np.ascontiguousarray(w.indices)).to(dev)
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    dq = torch.empty((T, H, 576), dtype=torch.bfloat16, device=dev)
    dkv32 = torch.empty((T, 1, 576), dtype=torch.float32, device=dev)
    dkv = torch.empty((T, 1, 576), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(capi.sparse_mla_bwd_workspace_bytes(T, H, topk, 0), 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for k in range(warmup + steps):
        flush.zero_()
        if k >= warmup:
            ev[k - warmup][0].record(stream)
        capi.sparse_mla_fwd(q, kv, idx, cu, w.scale, out=out, lse=lse)
        if k >= warmup:
            ev[k - warmup][1].record(stream)
        capi.sparse_mla_bwd(q, kv, out, dout, lse, idx, cu, w.scale, dq=dq, dkv_f32=dkv32, dkv=dkv, workspace=ws)
        if k >= warmup:
            ev[k - warmup][2].record(stream)
    torch.cuda.synchronize()
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    bwd_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    finite = bool(torch.isfinite(lse).all()) and bool(torch.isfinite(dkv32).all()) and \
        bool(torch.isfinite(dq.float()).all()) and bool(torch.isfinite(out.float()).all())
    fwd_flop = FWD_FLOP_PER_SLOT_HEAD * H * n_valid
    bwd_flop = BWD_FLOP_PER_SLOT_HEAD * H * n_valid
    gbytes = GATHER_BYTES_PER_SLOT * n_valid
    tp = peaks["bf16_tflops_sustained"]
    hbm = peaks["hbm_gbs"]

    def bound_ms(flop):
        return max(flop / (tp * 1e12), gbytes / (hbm * 1e9)) * 1e3

    def leg(ms, flop):
        b = bound_ms(flop)
        return {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12, "tokens_per_s": T / (ms * 1e-3),
                "roofline_frac": b / ms, "bound_ms": b,
                "bound": "tensor" if flop / (tp * 1e12) > gbytes / (hbm * 1e9) else "gathered bytes at HBM",
                "gathered_kv_gbs": gbytes / (ms * 1e-3) / 1e9}

    res = {"workload": w.name, "T": T, "H": H, "topk": topk, "valid_slots": n_valid, "steps": steps,
           "fwd": leg(fwd_ms, fwd_flop), "bwd": leg(bwd_ms, bwd_flop),
           "tokens_per_s": T / ((fwd_ms + bwd_ms) * 1e-3), "outputs_finite": finite}
    del q, kv, dout, idx, cu, out, lse, dq, dkv32, dkv, ws, flush
    torch.cuda.empty_cache()
    return res


def traffic_record():
    """Per-launch DRAM traffic of the backward call from a committed ncu
    summary, used only if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
        if rec.get("source_hash") != kernel_source_hash():
            return None
        return rec
    except Exception:
        return None


# sources of the backward kernel whose DRAM traffic the record holds
TRAFFIC_SOURCES = ("tc_bwd.cu", "tc_common.cuh", "smla_common.cuh")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bwd_sparse_mla_gb300", "csrc")
    for f in TRAFFIC_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


E2E_CHUNKS = 16


def e2e_ranges(T: int, chunks: int = E2E_CHUNKS):
    """Row ranges of the streamed step: E2E_CHUNKS equal ranges, except that the
    first and the last are split into ranges of 1/8, 1/4 and 1/2 of a chunk (growing
    at the start, shrinking at the end), so that less of the first upload and of the
    last download is left outside the overlap."""
    c = T / chunks
    sizes = [c / 8, c / 8, c / 4, c / 2] + [c] * (chunks - 2) + [c / 2, c / 4, c / 8, c / 8]
    bounds, acc = [0], 0.0
    for x in sizes:
        acc += x
        bounds.append(min(T, round(acc)))
    bounds[-1] = T
    return [(bounds[i], bounds[i + 1] - bounds[i]) for i in range(len(sizes)) if bounds[i + 1] > bounds[i]]


def same_results(host, device, dev, rows=4096):
    """The streamed step's host results against the device-resident step's (same
    inputs): out, lse and dq bit for bit; dkv, the bf16 of an fp32 sum taken in
    another order, within one bf16 step.  Compared in slices of rows."""
    import torch
    ok = True
    for i, (h, d) in enumerate(zip(host, device)):
        for r0 in range(0, d.shape[0], rows):
            a, b = h[r0:r0 + rows].to(dev), d[r0:r0 + rows]
            if i < 3:
                ok &= bool(torch.equal(a, b))
            else:
                a, b = a.float(), b.float()
                floor = 1e-5 * float(b.abs().max()) + 1e-30      # sums that cancel to near zero
                ok &= bool(((a - b).abs() <= b.abs() * 2.0 ** -7 + floor).all())
    return ok


def run_e2e(args, capi, w, dev, h_q, h_kv, h_dout, h_idx, h_cu):
    """Same step through the public API from pinned host buffers: H2D of the
    inputs, forward, backward, D2H of out, lse, dq and dkv (bf16), all inside the
    timed region.  The step streams through the device in E2E_CHUNKS ranges of
    query rows (sparse_mla_fwd_rows / sparse_mla_bwd_rows / sparse_mla_dkv_cast),
    each range's forward followed by its backward: a range starts as soon as its
    q and indices have landed, its dO uploads while its forward runs, its out /
    lse and dq download while later ranges compute, and dkv (fp32, accumulated
    over all ranges) is cast and downloaded last.  Copies run on their own
    streams, so uploads and downloads keep pace with the ranges' compute."""
    import torch
    T, H, topk = w.T, w.H, w.topk
    pin = lambda t: t.pin_memory()  # noqa: E731
    hq, hkv, hdo, hidx, hcu = pin(h_q), pin(h_kv), pin(h_dout), pin(h_idx), pin(h_cu)
    o_out = torch.empty((T, H, 512), dtype=torch.bfloat16, pin_memory=True)
    o_lse = torch.empty((T, H), dtype=torch.float32, pin_memory=True)
    o_dq = torch.empty((T, H, 576), dtype=torch.bfloat16, pin_memory=True)
    o_dkv = torch.empty((T, 1, 576), dtype=torch.bfloat16, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hkv, hdo, hidx, hcu))
    d2h = sum(t.numel() * t.element_size() for t in (o_out, o_lse, o_dq, o_dkv))
    # device buffers, allocated once outside the timed region
    d_q, d_kv, d_do = (torch.empty_like(t, device=dev) for t in (hq, hkv, hdo))
    d_idx, d_cu = torch.empty_like(hidx, device=dev), torch.empty_like(hcu, device=dev)
    d_out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    d_lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    d_dq = torch.empty((T, H, 576), dtype=torch.bfloat16, device=dev)
    d_dkv32 = torch.empty((T, 1, 576), dtype=torch.float32, device=dev)
    d_dkv = torch.empty((T, 1, 576), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(capi.sparse_mla_bwd_workspace_bytes(T, H, topk), 256), dtype=torch.uint8, device=dev)
    cs = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    # ranges alternate between two compute streams: they are independent (their dKV
    # contributions add commutatively), so one range's tail overlaps the next one's work
    comp = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
    ranges = e2e_ranges(T)

    def one(start):
        ev = lambda: torch.cuda.Event()  # noqa: E731
        ev_meta, ev_zero, ev_cast, ev_done = ev(), ev(), ev(), ev()
        ev_q, ev_do, ev_f, ev_b = ([ev() for _ in ranges] for _ in range(4))
        s_in.wait_event(start)
        with torch.cuda.stream(s_in):
            d_kv.copy_(hkv, non_blocking=True)
            d_cu.copy_(hcu, non_blocking=True)
            ev_meta.record(s_in)
            for c, (t0, nt) in enumerate(ranges):      # range by range: q, indices, then dO
                d_q[t0:t0 + nt].copy_(hq[t0:t0 + nt], non_blocking=True)
                d_idx[t0:t0 + nt].copy_(hidx[t0:t0 + nt], non_blocking=True)
                ev_q[c].record(s_in)
                d_do[t0:t0 + nt].copy_(hdo[t0:t0 + nt], non_blocking=True)
                ev_do[c].record(s_in)
        cs.wait_event(start)
        d_dkv32.zero_()                                # the row-range backward adds into it
        ev_zero.record(cs)
        for c, (t0, nt) in enumerate(ranges):          # each range's forward, then its backward
            st = comp[c % 2]
            st.wait_event(ev_meta)
            st.wait_event(ev_q[c])
            capi.sparse_mla_fwd_rows(d_q, d_kv, d_idx, d_cu, w.scale, t0, nt, d_out, d_lse, stream=st)
            ev_f[c].record(st)
            st.wait_event(ev_do[c])
            st.wait_event(ev_zero)
            capi.sparse_mla_bwd_rows(d_q, d_kv, d_out, d_do, d_lse, d_idx, d_cu, w.scale, t0, nt, d_dq, d_dkv32, ws,
                                     stream=st)
            ev_b[c].record(st)
        for c in range(len(ranges)):
            cs.wait_event(ev_b[c])
        capi.sparse_mla_dkv_cast(d_dkv32, d_dkv)
        ev_cast.record(cs)
        with torch.cuda.stream(s_out):
            for c, (t0, nt) in enumerate(ranges):
                s_out.wait_event(ev_f[c])
                o_out[t0:t0 + nt].copy_(d_out[t0:t0 + nt], non_blocking=True)
                o_lse[t0:t0 + nt].copy_(d_lse[t0:t0 + nt], non_blocking=True)
                s_out.wait_event(ev_b[c])
                o_dq[t0:t0 + nt].copy_(d_dq[t0:t0 + nt], non_blocking=True)
            s_out.wait_event(ev_cast)
            o_dkv.copy_(d_dkv, non_blocking=True)
            ev_done.record(s_out)
        cs.wait_event(ev_done)

    warm = torch.cuda.Event()
    warm.record(cs)
    one(warm)
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, args.e2e_steps))
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cs)
        one(a)
        b.record(cs)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = float(np.mean(times))
    # the streamed step's results against the device-resident step (same inputs): out, lse and dq bit
    # for bit, dkv (bf16 of an fp32 sum in another order) within one bf16 step
    return {"value": T / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": steps, "chunks": len(ranges), "dkv_mode": "atomic",
            "overlap": f"streamed in {len(ranges)} ranges of query rows (tapered at both ends) on two alternating "
                       "compute streams, each range's forward then backward: a range's q / indices / dO upload and "
                       "its out / lse / dq download overlap other ranges' work (separate copy streams)",
            "_host": (o_out, o_lse, o_dq, o_dkv)}


def run_topk(args):
    """Times the top-k index selection (sparse_mla_topk) alone on the workload's
    sequence layout: seeded N(0,1) fp32 index scores [T, longest sequence],
    each row reading its causal candidates; prints one JSON line (not the
    step's line).  Its bound is HBM: every candidate score is read once."""
    import torch
    from bwd_sparse_mla_gb300 import capi
    dev = torch.device("cuda", 0)
    capi.load()
    w = W.make_workload(args.config, values=False)
    cu_np = np.asarray(w.cu_seqlens, dtype=np.int64)
    if args.tokens:
        T = min(args.tokens, w.T)
        cu_np = np.minimum(cu_np, T)
        cu_np = np.unique(cu_np)
    else:
        T = w.T
    ncols = int(np.diff(cu_np).max())
    cand = int(sum(min(p + 1, ncols) for s0, s1 in zip(cu_np[:-1], cu_np[1:]) for p in range(s1 - s0)))
    cu = torch.from_numpy(cu_np.astype(np.int32)).to(dev)
    g = torch.Generator(device=dev).manual_seed(0)
    scores = torch.randn(T, ncols, device=dev, generator=g)
    idx = torch.empty((T, 1, w.topk), dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        capi.sparse_mla_topk(scores, cu, w.topk, indices=idx)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        capi.sparse_mla_topk(scores, cu, w.topk, indices=idx)
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = float(np.mean(times))
    peaks, src = load_peaks()
    gbs = cand * 4 / (ms * 1e-3) / 1e9
    print(json.dumps({
        "kernel": "sparse_mla_topk", "workload": w.name, "rows": T, "ncols": ncols, "topk": w.topk,
        "candidates": cand, "ms": ms, "steps": args.steps, "warmup": args.warmup,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "peak_source": src,
                     "algorithmic_bytes": cand * 4},
        "l2": "flushed before every timed call (256 MiB write)"}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5, help="workload 1..5 (5 = headline)")
    ap.add_argument("--tokens", type=int, default=0, help="use only the first N tokens (small profiling case)")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--workloads", default="1,2,3,4",
                    help="other workloads timed after the headline (comma list of 1..4, or 'none')")
    ap.add_argument("--workload-steps", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-rows", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dkv-mode", type=int, default=0, choices=[0, 1],
                    help="dKV accumulation of the timed backward: 0 = fp32 atomics, 1 = sorted segmented reduction")
    ap.add_argument("--other-mode-steps", type=int, default=2,
                    help="after the timed region, time the backward in the other dKV mode for this many steps")
    ap.add_argument("--clocks-csv", default=None,
                    help="also write the nvidia-smi clock samples of the timed region to this CSV file")
    ap.add_argument("--topk-only", action="store_true",
                    help="time only the top-k index selection on the workload's sequence layout")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.topk_only:
        run_topk(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
