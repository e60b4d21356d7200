"""Host-side logic of bench.py that needs no GPU: the recorded DRAM traffic is
used only while the kernel sources are unchanged, the roofline peaks come from
MEASURED_PEAKS.json when present (else the labelled fallback), and the L2 flush
writes then reads back."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    csrc = tmp_path / "int8_qmv_qmm_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.QMV_SOURCES:
        (csrc / name).write_text(f"// {name}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _write_profile(root, traffic, sha):
    (root / "profiles" / "p.txt").write_text(
        f"some notes\ntraffic_bytes_per_launch: {traffic}\nsource_sha256: {sha}\n")


def test_traffic_is_used_while_the_sources_match(fake_root):
    _write_profile(fake_root, 12345, bench.sources_sha256(bench.QMV_SOURCES))
    assert bench.profile_traffic("p.txt", bench.QMV_SOURCES) == 12345.0


def test_traffic_is_dropped_once_a_source_changes(fake_root):
    _write_profile(fake_root, 12345, bench.sources_sha256(bench.QMV_SOURCES))
    (fake_root / "int8_qmv_qmm_gb300" / "csrc" / "qmv_core.cuh").write_text("// changed\n")
    assert bench.profile_traffic("p.txt", bench.QMV_SOURCES) is None


def test_traffic_missing_or_malformed_is_none(fake_root):
    assert bench.profile_traffic("absent.txt", bench.QMV_SOURCES) is None
    _write_profile(fake_root, "not-a-number", bench.sources_sha256(bench.QMV_SOURCES))
    assert bench.profile_traffic("p.txt", bench.QMV_SOURCES) is None


def test_peaks_fall_back_and_say_so(fake_root):
    p = bench.load_peaks()
    assert p["source"] == "fallback"
    assert p["hbm_gbs"] == bench.FALLBACK_PEAKS["hbm_gbs"]


def test_peaks_measured_when_the_file_is_there(fake_root):
    (fake_root / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6687.8, "bf16_tflops": 1920.0, "bf16_tflops_sustained": 1727.7}))
    p = bench.load_peaks()
    assert p["source"] == "measured"
    assert (p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"]) == (6687.8, 1920.0, 1727.7)


def test_peaks_incomplete_file_falls_back(fake_root):
    (fake_root / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6687.8}))
    assert bench.load_peaks()["source"] == "fallback"


def test_flush_writes_then_reads(monkeypatch):
    import torch
    buf = torch.zeros(1024)
    bench.flush_l2(buf)
    assert torch.all(buf == 1.0)
