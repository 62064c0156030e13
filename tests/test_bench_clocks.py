"""Host-side parsing of the bench's clock samples (nvidia-smi CSV lines): the
median SM clock under load, the highest maximum clock and every throttle
reason seen active; unparsable lines are skipped."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def summary_of(lines):
    c = bench.ClockSampler(-1)
    c.lines = lines
    return c.summary()


def test_reasons_clock_and_power():
    s = summary_of([
        "1650, 2070, 1398.5, 0x4, Not Active, Not Active, Not Active, Active",
        "1610, 2070, 1401.0, 0x4, Not Active, Not Active, Not Active, Active",
        "1700, 2070, 1395.0, 0x0, Not Active, Not Active, Active, Not Active",
        "garbage",
        "[N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1650.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]


def test_no_samples():
    s = summary_of([])
    assert s["samples"] == 0 and s["reasons"] == ["not sampled"]
