"""Host logic of bench.py that needs no GPU: the clock record keeps only the
nvidia-smi samples inside the timed region and reports throttle reasons."""
import datetime
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sampler(n, cap_at=None, slow_from=None):
    c = bench.ClockSampler(0)
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)
    for i in range(n):
        ts = (base + datetime.timedelta(milliseconds=50 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        sm = 1800 if slow_from is not None and i >= slow_from else 2070
        cap = "Active" if i == cap_at else "Not Active"
        c.lines.append(f"{ts}, {sm}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}")
    return c, (lambda ms: (base + datetime.timedelta(milliseconds=ms)).timestamp())


def test_clock_summary_keeps_the_timed_window():
    c, t = _sampler(10, cap_at=7, slow_from=6)
    s = c.summary(t(120), t(380))  # samples at 150 .. 350 ms
    assert s["samples"] == 5 and s["window"] == "inside the timed region"
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    s = c.summary(t(0), t(120))  # samples at 0 .. 100 ms: no reason there
    assert s["samples"] == 3 and s["reasons"] == []


def test_clock_summary_short_region_takes_the_next_sample():
    c, t = _sampler(4)
    s = c.summary(t(10), t(40))
    assert s["samples"] == 1 and "none inside" in s["window"]


def test_clock_summary_without_samples_is_none():
    assert bench.ClockSampler(0).summary(0.0, 1.0) is None
