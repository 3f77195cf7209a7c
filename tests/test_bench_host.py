"""Host logic of bench.py that needs no GPU: the clock record of the timed
region (nvidia-smi samples filtered to the region's wall-clock window)."""
import datetime
import os
import tempfile

import bench


def _line(t, mhz, power, power_cap="Not Active", hw="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, 0, {mhz}, 2070, {power}, {hw}, Not Active, Not Active, {power_cap}\n"


def _sampler(lines):
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.writelines(lines)
    c.proc = object()  # a sampler that ran
    return c


def test_clock_summary_keeps_only_samples_inside_the_timed_region():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.2, 2070, 170.0),                      # before: idle
             _line(t0 + 0.02, 1900, 400.0),
             _line(t0 + 0.04, 1790, 800.0, power_cap="Active"),
             _line(t0 + 0.06, 1800, 900.0, power_cap="Active"),
             _line(t0 + 0.5, 300, 150.0, hw="Active")]           # after: idle, throttled
    c = _sampler(lines)
    c.mark(t0, t0 + 0.1)
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1800 and s["sm_mhz_min"] == 1790
    assert s["reasons"] == ["sw_power_cap"]       # hw_slowdown was outside the region
    assert s["power_w_max"] == 900.0


def test_clock_summary_without_samples_in_the_region_says_so():
    t0 = 1_800_000_000.0
    c = _sampler([_line(t0 - 1.0, 2070, 170.0)])
    c.mark(t0, t0 + 0.01)
    s = c.summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None
    assert s["reasons"] == ["no samples inside the timed region"]
