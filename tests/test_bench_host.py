"""bench.py's host-side helpers on CPU: the clock record taken during the
timed region (median SM clock, the maximum, and which throttle reasons were
active) and the roofline denominators (the measured peaks, else the fallback)."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

IDLE = "2070, 2070, 310.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
CAPPED = "1965, 2070, 1398.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
HOT = "1410, 2070, 1100.0, 0x0000000000000008, Active, Not Active, Not Active, Not Active"


def summary_of(lines):
    cs = bench.ClockSampler(0)
    cs.out = "\n".join(lines) + "\n"
    return cs.summary()


def test_median_clock_and_active_reasons():
    s = summary_of([IDLE, CAPPED, IDLE, IDLE, CAPPED])
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 5}


def test_hw_slowdown_is_reported():
    s = summary_of([IDLE, HOT, HOT])
    assert s["reasons"] == ["hw_slowdown"] and s["sm_mhz"] == 1410.0


def test_malformed_and_missing_samples():
    s = summary_of(["[N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]", "garbage", IDLE])
    assert s["samples"] == 1 and s["sm_mhz"] == 2070.0
    empty = bench.ClockSampler(0)
    empty.out = ""
    assert empty.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_peaks_come_from_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (6800.0, 1900.0, 1700.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6689.1, "bf16_tflops": 1941.1,
                                                               "bf16_tflops_sustained": 1735.0}))
    assert bench.peaks() == (6689.1, 1941.1, 1735.0, "measured")
