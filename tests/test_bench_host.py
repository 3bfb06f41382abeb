"""Host-side pieces of bench.py that need no GPU: the clock sampler's parsing
and window selection, the code-only kernel hash, the peak selection and the
traffic lookup keyed to that hash."""
import json
import os

import pytest

import bench


def _write_samples(path, rows):
    with open(path, "w") as fh:
        for ts, clk, power, power_cap in rows:
            fh.write(f"{ts}, 0, {clk}, 2070, {power}, 0x0, Not Active, Not Active, Not Active, "
                     f"{'Active' if power_cap else 'Not Active'}\n")


def test_clock_summary_keeps_the_timed_window(tmp_path):
    c = bench.ClockSampler(0)
    c.path = str(tmp_path / "clocks.csv")
    _write_samples(c.path, [
        ("2026/12/02 10:00:00.000", 2070, 300.0, False),    # before the window
        ("2026/12/02 10:00:00.500", 1600, 1380.0, True),
        ("2026/12/02 10:00:00.600", 1650, 1390.0, True),
        ("2026/12/02 10:00:00.700", 1700, 1370.0, True),
        ("2026/12/02 10:00:01.500", 2070, 250.0, False),    # after it
    ])
    c.mark(c._epoch("2026/12/02 10:00:00.450"), c._epoch("2026/12/02 10:00:00.750"))
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1650 and s["sm_min_mhz"] == 1600
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_median"] == 1380.0


def test_clock_summary_falls_back_to_the_nearest_samples(tmp_path):
    c = bench.ClockSampler(0)
    c.path = str(tmp_path / "clocks.csv")
    _write_samples(c.path, [("2026/12/02 10:00:00.000", 1900, 900.0, False),
                            ("2026/12/02 10:00:00.100", 1800, 1000.0, True),
                            ("2026/12/02 10:00:05.000", 2070, 200.0, False)])
    c.mark(c._epoch("2026/12/02 10:00:00.120"), c._epoch("2026/12/02 10:00:00.130"))
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 1850.0


def test_clock_summary_without_samples(tmp_path):
    c = bench.ClockSampler(0)
    c.path = str(tmp_path / "missing.csv")
    assert c.summary()["samples"] == 0


def test_code_hash_ignores_comments_and_whitespace():
    a = "int f(int x) {  // doubles x\n  return 2 * x; /* fast */ }\n"
    b = "/* a new comment */\nint f(int x) {\n\n  return 2 * x;\n}  // trailing\n"
    c = "int f(int x) { return 3 * x; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_peaks_read_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks()[3] == "fallback"
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6500.0}))
    burst, sustained, hbm, kind = bench.peaks()
    assert (burst, sustained, hbm, kind) == (1900.0, 1700.0, 6500.0, "measured")


def test_roofline_peak_follows_the_timed_window():
    # a short window (20 steps of about 7 ms) is a burst; seconds of steps run
    # into the power cap like the sustained measurement
    peak, desc = bench.roofline_peak(0.135, 1942.5, 1708.6, "measured")
    assert peak == 1942.5 and "burst" in desc
    peak, desc = bench.roofline_peak(bench.SUSTAINED_WINDOW_S, 1942.5, 1708.6, "measured")
    assert peak == 1708.6 and "sustained" in desc


def test_traffic_is_reported_only_for_the_captured_code(tmp_path, monkeypatch):
    kh = bench.kernel_hash()
    f = tmp_path / "ncu_traffic.txt"
    f.write_text("# comment\n"
                 f"kernel_hash={kh} workload=w1 gemm_bytes_per_launch=1.5e9 source=x\n"
                 "kernel_hash=0000000000000000 workload=w2 gemm_bytes_per_launch=2.5e9 source=x\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.measured_traffic("w1") == 1.5e9
    assert bench.measured_traffic("w2") is None
    assert bench.measured_traffic("w3") is None

