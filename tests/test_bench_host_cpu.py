"""Host-side helpers of bench.py on CPU: the clock summary taken from nvidia-smi rows
(median SM clock inside the timed window, throttle reasons seen, fallback to the whole
run when no sample falls inside), the DRAM-traffic record that is reported only for
the kernel source it was captured from, and the measured-peak lookup."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

pytest.importorskip("torch")
import bench  # noqa: E402


def _row(mhz, mx=2070, reasons=("Not Active",) * 4):
    return "2026/12/02 10:00:00.000, %d, %d, 900.00, 0x0, %s" % (mhz, mx, ", ".join(reasons))


def test_clock_summary_inside_the_window():
    s = bench.ClockSampler(0)
    s.rows = [(1.0, _row(1000)), (2.0, _row(2070)), (2.5, _row(2055)),
              (3.0, _row(2070, reasons=("Not Active", "Not Active", "Not Active", "Active"))),
              (9.0, _row(500))]
    out = s.summary(1.5, 3.5)
    assert out["window"] == "timed" and out["samples"] == 3
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_falls_back_to_the_run_and_skips_bad_rows():
    s = bench.ClockSampler(0)
    s.rows = [(1.0, _row(1900)), (2.0, "garbage"), (3.0, "a, b, c, d, e, f, g, h, i"),
              (4.0, _row(2000, reasons=("Active", "Not Active", "Active", "Not Active")))]
    out = s.summary(10.0, 11.0)
    assert out["window"] == "run" and out["samples"] == 2
    assert out["sm_mhz"] == 1950
    assert out["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    empty = bench.ClockSampler(0).summary(0.0, 1.0)
    assert empty["samples"] == 0 and empty["sm_mhz"] is None


def test_traffic_record_only_for_its_own_source():
    rec = json.load(open(os.path.join(ROOT, "profiles", "ssd_stream_kernel_c5_traffic.json")))
    assert rec["passes"] == 1
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert rec["dram_bytes_read"] >= rec["algorithmic_bytes_per_launch"]
    assert bench.traffic_record(rec["source_digest"]) == rec["dram_bytes_per_launch"]
    assert bench.traffic_record("0" * 16) is None


def test_measured_peak_source():
    peak, kind = bench.measured_peak()
    assert peak > 0
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured"
    else:
        assert kind == "fallback" and peak == bench.FALLBACK_HBM_GBS
