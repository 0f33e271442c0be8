"""The benchmark's clock record: nvidia-smi rows are read with their
timestamps, only the rows stamped inside the timed region count (the nearest
later row when the region is shorter than the sampling period), and any
throttle reason seen there is reported.  Host logic only: the rows below are
written by the test, nothing runs on a GPU."""
import datetime
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

T = time.time()


def _row(dt, mhz, power_cap="Not Active", thermal="Not Active"):
    ts = datetime.datetime.fromtimestamp(T + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, 0, {mhz}, 2070, 812.5, 0x0, Not Active, {thermal}, Not Active, {power_cap}"


ROWS = [_row(-0.50, 1200), _row(0.004, 2040), _row(0.014, 1980, power_cap="Active"), _row(0.024, 2070),
        _row(0.30, 2070, thermal="Active")]


def test_only_rows_inside_the_region_count():
    s = bench.ClockSampler.summarize(bench.ClockSampler.parse(ROWS), (T, T + 0.03))
    assert s["samples_in_timed_region"] == 3 and s["samples"] == 3
    assert s["sm_mhz"] == 2040 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]  # the idle row before and the thermal row after are outside


def test_region_shorter_than_the_period_takes_the_next_row():
    s = bench.ClockSampler.summarize(bench.ClockSampler.parse(ROWS), (T + 0.025, T + 0.028))
    assert s["samples_in_timed_region"] == 0 and s["samples"] == 1
    assert s["sm_mhz"] == 2070 and s["reasons"] == ["hw_thermal_slowdown"]


def test_malformed_rows_are_skipped_and_no_rows_is_reported():
    rows = bench.ClockSampler.parse(["", "garbage", "a, b, c"])
    assert rows == []
    s = bench.ClockSampler.summarize(rows, (T, T + 1))
    assert s["samples"] == 0 and s["sm_mhz"] is None
