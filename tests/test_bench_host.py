"""Host-side pieces of bench.py, on CPU: the committed DRAM-traffic records are
used only while every kernel source they list is unchanged, the peaks fall back
when the measured file is missing, and the clock sampler's parsing reports the
throttle reasons that make a run invalid and the median clock under load.
"""
import hashlib
import json
import os
import shutil

from conftest import ROOT

import bench

SOURCES = ["chunked_prefill_mixed_decode_gb300/csrc/attention.cu",
           "chunked_prefill_mixed_decode_gb300/csrc/append_rope.cuh"]


def _tree(tmp_path, shas=None):
    """A copy of the kernel sources and one traffic record under tmp_path."""
    for src in SOURCES:
        dst = tmp_path / src
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copyfile(os.path.join(ROOT, src), dst)
    if shas is None:
        shas = {src: hashlib.sha256((tmp_path / src).read_bytes()).hexdigest() for src in SOURCES}
    (tmp_path / "profiles").mkdir(exist_ok=True)
    rec = {"kernel": "attention_kernel", "workload": "w", "batch": 0, "sources": shas,
           "dram_bytes_read": 1000, "dram_bytes_write": 10, "append_dram_bytes": 5}
    (tmp_path / "profiles" / "attention_kernel_w.traffic.json").write_text(json.dumps(rec))
    return rec


def test_traffic_record_is_used_while_its_sources_match(tmp_path, monkeypatch):
    rec = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    got = bench.captured_traffic("w")
    assert got is not None and got["dram_bytes_read"] == rec["dram_bytes_read"]
    assert bench.captured_traffic("missing") is None


def test_traffic_record_is_dropped_when_a_kernel_changes(tmp_path, monkeypatch):
    _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    with open(tmp_path / SOURCES[1], "a") as f:
        f.write("\n// edited\n")
    assert bench.captured_traffic("w") is None


def test_traffic_record_with_a_missing_source_is_dropped(tmp_path, monkeypatch):
    _tree(tmp_path, shas={"no/such/file.cu": "0" * 64})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.captured_traffic("w") is None


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.read_peaks()
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6000, "bf16_tflops": 1800}))
    peaks, src = bench.read_peaks()
    assert src == "measured" and peaks["hbm_gbs"] == 6000.0
    assert peaks["bf16_tflops_sustained"] == 1800.0  # no sustained figure: the burst one


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampled(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.fh = open(os.devnull, "w")
    s.proc = _Done()
    return s.stop()


def test_clock_sampler_reports_throttle_reasons_and_median_under_load(tmp_path):
    # index, sm MHz, max MHz, power W, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    lines = ["0, 1000, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1950, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2000, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    c = _sampled(tmp_path, lines)
    assert c["sm_mhz"] == 2000.0  # median of the samples above 200 W
    assert c["sm_max_mhz"] == 2070.0 and c["samples"] == 4
    assert c["reasons"] == ["sw_power_cap"]
    lines[1] = "0, 1400, 2070, 900.0, 0x40, Active, Not Active, Active, Not Active"
    c = _sampled(tmp_path, lines)
    assert c["reasons"] == sorted(["hw_slowdown", "sw_thermal_slowdown", "sw_power_cap"])


def test_clock_sampler_without_samples_says_so(tmp_path):
    c = _sampled(tmp_path, ["garbage line"])
    assert c["reasons"] == ["unsampled"] and c["sm_mhz"] is None
