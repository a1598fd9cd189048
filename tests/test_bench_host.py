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


def test_step_roofline_terms_and_overlap_bound():
    import synth
    dims = synth.MISTRAL_LAYER
    ctxs = [128, 4096, 1000]
    per_op, overlap, ops, t_math, t_mem = bench.step_roofline(dims, ctxs, 8000.0, 2000.0)
    # QKV: 2 * 512 * 4096 * 6144 flops at 2000 TFLOP/s (math-bound at 512 rows)
    assert abs(ops["gemm_qkv"] - 2 * 512 * 4096 * 6144 / 2e15) < 1e-12
    # decode attention: every key and value once + q/out rows at 8000 GB/s (memory-bound)
    kv = sum(c + 1 for c in ctxs) * 8 * 128 * 2 * 2 + 3 * 4096 * 2 * 2
    assert abs(ops["decode_attn"] - kv / 8e12) < 1e-12
    # chunk attention averaged over the three starts: keys of query i at start s are s + i + 1
    want = sum(4 * 128 * 32 * sum(s + i + 1 for i in range(448)) for s in (0, 512, 1536)) / 3 / 2e15
    assert abs(ops["chunk_attn"] - want) < 1e-12  # math-bound: its keys are a few MB
    assert abs(per_op - sum(ops.values())) < 1e-15
    assert overlap == max(t_math, t_mem) and overlap <= per_op


def test_traffic_is_null_once_the_kernel_source_changed(monkeypatch):
    t = dict(bench.TRAFFIC["decode_attn"])
    monkeypatch.setitem(bench.TRAFFIC, "decode_attn", dict(t, sha=bench.source_sha(t["files"])))
    val, src = bench.traffic_of("decode_attn")
    assert val == t["bytes"] and "ncu capture" in src
    monkeypatch.setitem(bench.TRAFFIC, "decode_attn", dict(t, sha="0" * 16))
    val, src = bench.traffic_of("decode_attn")
    assert val is None and "changed" in src
    assert bench.traffic_of("gemm_o")[0] is None
