"""Host-side pieces of bench.py that need no GPU: the clock-sample parser
keeps the nvidia-smi samples taken inside the timed region, the roofline's
DRAM traffic comes only from a profile of the current kernel source, and the
HBM peak is the measured one when it is there."""
import datetime
import hashlib
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


def test_profiled_traffic_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    """The roofline's DRAM traffic comes from a committed ncu summary, and only
    while the kernel source still hashes to the value recorded in it."""
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_bytes(b"kernel, first version")
    sha = hashlib.sha256(b"kernel, first version").hexdigest()
    (tmp_path / "profiles" / "p.md").write_text(
        "| metric | value |\n|---|---|\n\n"
        "- traffic_bytes_per_launch: 1234567\n"
        "- algorithmic bytes per launch: 1,200,000\n"
        f"- source_sha256: {sha}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("p.md", "k.cu") == 1234567
    src.write_bytes(b"kernel, second version")
    assert bench.profiled_traffic("p.md", "k.cu") is None
    assert bench.profiled_traffic("absent.md", "k.cu") is None


def test_peaks_prefers_the_measured_file(tmp_path, monkeypatch):
    """The HBM denominator is the measured copy bandwidth when the file is
    there, else the stated fallback."""
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6000.5}')
    assert bench.peaks() == (6000.5, "measured")
