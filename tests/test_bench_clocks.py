"""The benchmark's clock summary (host logic, no GPU): nvidia-smi samples
taken during the timed region become the median SM clock, the maximum clock,
the throttle reasons seen and, when the region held at least 20 samples, the
median board power."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, power, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active"):
    return f"{sm}, 2070, {power}, 0x0, {hw}, {hw_th}, {sw_th}, {cap}"


def _summary(lines):
    c = bench.ClockSampler(0)
    c.lines = list(lines)
    return c.summary()


def test_median_clock_max_clock_and_power_under_load():
    lines = [_line(1600 + i, 1300.0 + i, cap="Active") for i in range(25)]
    s = _summary(lines)
    assert s["sm_mhz"] == 1612 and s["sm_max_mhz"] == 2070 and s["samples"] == 25
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w"] == 1312.0


def test_short_region_reports_no_power():
    s = _summary([_line(2070, 180.0) for _ in range(5)])
    assert s["sm_mhz"] == 2070 and "power_w" not in s and s["reasons"] == []


def test_every_throttle_reason_is_seen():
    lines = [_line(1500, 900.0, hw="Active"), _line(1500, 900.0, hw_th="Active"),
             _line(1500, 900.0, sw_th="Active"), _line(1500, 900.0, cap="Active"), _line(2070, 500.0)]
    s = _summary(lines)
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_malformed_and_missing_samples():
    s = _summary(["", "garbage", "1700, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active",
                  "[N/A], 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active"])
    assert s["samples"] == 1 and s["sm_mhz"] == 1700 and "power_w" not in s
    assert _summary([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
