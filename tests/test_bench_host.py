"""Host-side logic of bench.py that needs no GPU: the clock-sample summary that
decides whether a timed run is kept, the ncu traffic figure tied to the kernel
source it was taken on, and the roofline denominator."""
import hashlib
import json
import os

import pytest

import bench


def test_clock_summary_median_max_and_reasons():
    lines = [
        "2026/12/02 21:13:01.100, 2032, 2032, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 21:13:01.200, 1980, 2032, Not Active, Not Active, Not Active, Active",
        "2026/12/02 21:13:01.300, 2010, 2032, Not Active, Not Active, Not Active, Not Active",
    ]
    s = bench.summarize_clock_lines(lines)
    assert s["sm_mhz"] == 2010 and s["sm_max_mhz"] == 2032 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_names_every_slowdown_column():
    line = "2026/12/02 21:13:01.100, 1500, 2032, Active, Active, Active, Not Active"
    assert bench.summarize_clock_lines([line])["reasons"] == [
        "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_skips_malformed_lines():
    lines = ["garbage", "2026/12/02 21:13:01.100, [N/A], 2032, Not Active, Not Active, "
             "Not Active, Not Active", ""]
    s = bench.summarize_clock_lines(lines)
    assert s == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


@pytest.fixture
def tree(tmp_path, monkeypatch):
    csrc = tmp_path / "quantized_decode_attention_blocks_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _record(tree, src_text, entry):
    (tree / "quantized_decode_attention_blocks_b300" / "csrc" / "k.cu").write_text(src_text)
    with open(tree / "profiles" / "traffic.json", "w") as f:
        json.dump(entry, f)


def test_traffic_only_while_the_source_matches_the_capture(tree):
    src = "__global__ void k() {}\n"
    h = hashlib.sha256(src.encode()).hexdigest()[:16]
    _record(tree, src, {"k": {"dram_bytes_per_launch": 1234.0, "source_sha256_16": h,
                              "workload": "w1", "algorithmic_bytes_per_launch": 1000}})
    assert bench.ncu_traffic("k", "k.cu", "w1", 1000) == (1234.0, "ncu capture of w1")
    # any edit to the source since the capture: the figure no longer applies
    (tree / "quantized_decode_attention_blocks_b300" / "csrc" / "k.cu").write_text(src + " ")
    assert bench.ncu_traffic("k", "k.cu", "w1", 1000) == (None, None)
    assert bench.ncu_traffic("other", "k.cu", "w1", 1000) == (None, None)


def test_traffic_of_the_own_workload_else_scaled(tree):
    # the capture of the bench's workload is taken as it is; another
    # workload's is scaled by the ratio of algorithmic bytes per launch
    src = "__global__ void k() {}\n"
    h = hashlib.sha256(src.encode()).hexdigest()[:16]
    _record(tree, src, {
        "k": {"dram_bytes_per_launch": 950.0, "source_sha256_16": h, "workload": "small",
              "algorithmic_bytes_per_launch": 1000},
        "k@big": {"dram_bytes_per_launch": 3900.0, "source_sha256_16": h, "workload": "big",
                  "algorithmic_bytes_per_launch": 4000}})
    assert bench.ncu_traffic("k", "k.cu", "big", 4000) == (3900.0, "ncu capture of big")
    assert bench.ncu_traffic("k", "k.cu", "small", 1000) == (950.0, "ncu capture of small")
    b, src_note = bench.ncu_traffic("k", "k.cu", "third", 2000)
    assert b in (1900.0, 1950.0) and "scaled by" in src_note
    # a capture without its algorithmic bytes cannot be scaled: not used
    _record(tree, src, {"k": {"dram_bytes_per_launch": 950.0, "source_sha256_16": h,
                              "workload": "small"}})
    assert bench.ncu_traffic("k", "k.cu", "small", 1000) == (None, None)


def test_traffic_absent_without_a_record(tree):
    assert bench.ncu_traffic("k", "k.cu", "w1", 1000) == (None, None)


def test_peak_is_the_measured_copy_bandwidth_else_the_fallback(tree):
    assert bench.measured_peaks() == (6400.0, "fallback")
    with open(os.path.join(tree, "MEASURED_PEAKS.json"), "w") as f:
        json.dump({"hbm_gbs": 6479.9, "bf16_tflops": 1800.0}, f)
    assert bench.measured_peaks() == (6479.9, "measured")


def test_sampler_summarizes_only_the_timed_window():
    class _Proc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s = bench.ClockSampler()
    s.proc = _Proc()
    s.mark("t_start")
    s.mark("t_stop")
    t = s.t_start
    busy = "2026/12/02 21:13:01.100, 2032, 2032, Not Active, Not Active, Not Active, Active"
    idle = "2026/12/02 21:13:09.100, 345, 2032, Not Active, Not Active, Not Active, Not Active"
    s.lines = [(t - 5.0, idle), (t, busy), (t + 5.0, idle)]
    out = s.stop()
    assert out["samples"] == 1 and out["sm_mhz"] == 2032 and out["reasons"] == ["sw_power_cap"]
