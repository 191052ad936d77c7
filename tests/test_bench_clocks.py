"""Host logic of bench.py's clock record: parsing of nvidia-smi's CSV samples,
the timed-window filter and the throttle reasons (no GPU needed)."""
import os
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _line(t, mhz, reasons=("Not Active",) * 4):
    stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t)) + ".%03d" % int((t % 1) * 1000)
    return ", ".join([stamp, str(mhz), "2070", "700.00 W", "0x0", *reasons]) + "\n"


def _summary(lines, t0, t1):
    s = bench.ClockSampler(0)
    s.out.write("".join(lines))
    s.out.flush()
    return s.summary(t0, t1)


def test_samples_inside_the_window_only():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 1.0, 345)]  # idle, before the timed phase
    lines += [_line(t0 + 0.1 * i, 2070 - i) for i in range(6)]
    lines += [_line(t0 + 2.0, 345)]  # idle, after it
    out = _summary(lines, t0, t0 + 0.6)
    assert out["samples"] == 6 and out["window"] == "timed"
    assert out["sm_mhz"] == 2067.5 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == []


def test_throttle_reasons_are_reported():
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.1, 1900, ("Not Active", "Not Active", "Not Active", "Active")),
             _line(t0 + 0.2, 1800, ("Active", "Not Active", "Not Active", "Not Active"))]
    out = _summary(lines, t0, t0 + 0.3)
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_no_sample_in_the_window_falls_back_to_the_whole_run():
    t0 = 1_800_000_000.0
    out = _summary([_line(t0 - 5.0, 2070), "garbage line\n"], t0, t0 + 0.001)
    assert out["window"] == "whole run" and out["samples"] == 1


def test_no_samples_at_all():
    out = _summary([], 0.0, 1.0)
    assert out["samples"] == 0 and out["reasons"] == ["no samples"]
