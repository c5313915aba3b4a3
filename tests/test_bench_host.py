"""Host-side pieces of bench.py that need no GPU: the clock-sample parser
keeps the nvidia-smi samples taken inside the timed region."""
import datetime
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _line(t, mhz, power_cap="Not Active", thermal="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, 0, {mhz}, 2070, 950.0, 0x0, Not Active, Not Active, {thermal}, {power_cap}"


def test_clock_samples_inside_the_timed_window():
    now = time.time()
    text = "\n".join([
        _line(now - 1.0, 345),                          # idle, before the window
        _line(now + 0.1, 2070),
        _line(now + 0.3, 2055, power_cap="Active"),
        _line(now + 0.5, 2070),
        _line(now + 2.0, 990, thermal="Active"),        # after the window
    ])
    got = bench.Clocks.parse(text, [now, now + 0.6])
    assert got["samples"] == 3 and got["samples_in_timed_region"] == 3
    assert got["samples_total"] == 5
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]            # the thermal sample lies outside


def test_clock_samples_fall_back_to_all_when_none_inside():
    now = time.time()
    text = "\n".join([_line(now + 10.0, 2070), _line(now + 10.2, 2040)])
    got = bench.Clocks.parse(text, [now, now + 0.1])
    assert got["samples_in_timed_region"] == 0 and got["samples"] == 2
    assert got["sm_mhz"] == 2055.0


def test_clock_parser_ignores_garbage():
    assert bench.Clocks.parse("", None) is None
    assert bench.Clocks.parse("No devices were found\n", None) is None


def test_nvml_reason_bits_decode():
    assert bench.Clocks.decode(0) == set()
    assert bench.Clocks.decode(0x4) == {"sw_power_cap"}
    assert bench.Clocks.decode(0x1 | 0x8 | 0x40) == {"hw_slowdown", "hw_thermal_slowdown"}
    assert bench.Clocks.decode(0x20) == {"sw_thermal_slowdown"}


def test_sample_summary_window():
    now = time.time()
    samples = [(now - 1.0, 300.0, 2070.0, set()),
               (now + 0.01, 2070.0, 2070.0, set()),
               (now + 0.02, 2040.0, 2070.0, {"sw_power_cap"}),
               (now + 0.03, 2070.0, 2070.0, set())]
    got = bench.Clocks.summarize(samples, [now, now + 0.04])
    assert got["samples_in_timed_region"] == 3 and got["sm_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"] and got["samples_total"] == 4
    assert bench.Clocks.summarize([], None) is None
