"""bench.ClockSampler.summary on synthetic nvidia-smi lines (CPU only): the median SM clock under
load, the maximum clock, and which throttle reasons were active during the timed region ("Not
Active" must not count; malformed lines are skipped)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, mx, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return f"0, {sm}, {mx}, 950.12, 0x0000000000000000, {hw}, {hwt}, {swt}, {cap}"


def _summary(lines):
    s = bench.ClockSampler(0)
    s.lines = list(lines)
    return s.summary()


def test_median_max_and_no_reasons():
    got = _summary([_line(2032, 2032), _line(1980, 2032), _line(2010, 2032)])
    assert got == {"sm_mhz": 2010.0, "sm_max_mhz": 2032.0, "reasons": [], "samples": 3}


def test_active_reasons_are_reported_once_each():
    lines = [_line(1900, 2032, cap="Active"), _line(1850, 2032, cap="Active"),
             _line(1500, 2032, hwt="Active")]
    got = _summary(lines)
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert got["sm_mhz"] == 1850.0 and got["samples"] == 3


def test_malformed_lines_are_skipped():
    lines = ["", "[N/A]", "0, [N/A], 2032, 1, 0x0, Not Active, Not Active, Not Active, Not Active",
             _line(2032, 2032, hw="Active")]
    got = _summary(lines)
    assert got["samples"] == 1 and got["reasons"] == ["hw_slowdown"]


def test_no_samples():
    assert _summary([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
