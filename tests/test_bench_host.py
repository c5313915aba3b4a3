"""Host-side helpers of bench.py that decide what the JSON line reports."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


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
