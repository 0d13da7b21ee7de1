"""Host logic of the benchmark that needs no GPU: the roofline denominators
(measured peaks when the generated file is present, else the stated
fallback), the DRAM traffic record (used only while it matches the backward
kernel's sources) and the comparison of the streamed end-to-end step with the
device-resident one."""
import json
import os
import shutil

import pytest
import torch

import bench


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS


def test_measured_peaks_are_read_wherever_they_nest(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"gpu": "GB300", "peaks": {"hbm_gbs": 6692.8, "bf16_tflops": 1878.4, "bf16_tflops_sustained": 1701.0}}))
    peaks, src = bench.load_peaks()
    assert src == "measured"
    assert peaks == {"hbm_gbs": 6692.8, "bf16_tflops": 1878.4, "bf16_tflops_sustained": 1701.0}


def test_sustained_peak_defaults_to_the_burst_one(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0, "bf16_tflops": 1800.0}))
    peaks, src = bench.load_peaks()
    assert src == "measured" and peaks["bf16_tflops_sustained"] == 1800.0


def _copy_sources(tmp_path):
    csrc = tmp_path / "bwd_sparse_mla_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.TRAFFIC_SOURCES:
        shutil.copy(os.path.join(bench.ROOT, "bwd_sparse_mla_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    return csrc


def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    csrc = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"dram_bytes_per_launch": 123, "note": "n", "source_hash": bench.kernel_source_hash()}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.traffic_record()["dram_bytes_per_launch"] == 123
    with open(csrc / "tc_bwd.cu", "a") as f:            # the kernel changes: the counters no longer apply
        f.write("\n// changed\n")
    assert bench.traffic_record() is None


def test_committed_traffic_record_is_consistent():
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    assert rec["dram_bytes_per_launch"] == rec["dram_read_bytes"] + rec["dram_write_bytes"]
    assert set(rec["source_files"]) == set(bench.TRAFFIC_SOURCES)
    if rec["source_hash"] != bench.kernel_source_hash():
        # the benchmark then reports no traffic figure until the counters are taken again
        assert bench.traffic_record() is None
        pytest.skip("the backward kernel changed since its DRAM bytes were captured")


def test_streamed_results_are_compared_exactly_except_dkv():
    out = torch.randn(40, 2, 3).to(torch.bfloat16)
    lse = torch.randn(40, 2)
    dq = torch.randn(40, 2, 5).to(torch.bfloat16)
    dkv = torch.randn(40, 1, 5).to(torch.bfloat16)
    dev = "cpu"
    assert bench.same_results((out.clone(), lse.clone(), dq.clone(), dkv.clone()), (out, lse, dq, dkv), dev, rows=16)
    lse2 = lse.clone()
    lse2[33, 1] = torch.nextafter(lse2[33, 1], torch.tensor(1e9))    # one ulp in the last slice
    assert not bench.same_results((out, lse2, dq, dkv), (out, lse, dq, dkv), dev, rows=16)
    dkv2 = (dkv.float() * (1 + 2.0 ** -8)).to(torch.bfloat16)         # within one bf16 step
    assert bench.same_results((out, lse, dq, dkv2), (out, lse, dq, dkv), dev, rows=16)
    dkv3 = dkv.clone()
    dkv3[5, 0, 2] = dkv3[5, 0, 2] * 2 + 1                               # far off
    assert not bench.same_results((out, lse, dq, dkv3), (out, lse, dq, dkv), dev, rows=16)


@pytest.mark.parametrize("T", [1, 5, 17, 4096, 65536, 65537])
def test_streamed_ranges_partition_the_rows(T):
    r = bench.e2e_ranges(T)
    assert r[0][0] == 0 and sum(n for _, n in r) == T
    assert all(n > 0 for _, n in r)
    assert all(r[i][0] + r[i][1] == r[i + 1][0] for i in range(len(r) - 1))
    if T >= 16 * bench.E2E_CHUNKS:          # the edges taper: first and last ranges are the smallest
        sizes = [n for _, n in r]
        assert sizes[0] < max(sizes) and sizes[-1] < max(sizes)
