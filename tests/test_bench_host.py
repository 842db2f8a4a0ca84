"""Host-side logic of bench.py, without a GPU: the clock sampler's parsing of
nvidia-smi samples (through a stand-in nvidia-smi on PATH), and the guard that
only reports the committed DRAM traffic while the kernel source matches it."""
import os
import stat
import sys
import time
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
sys.path.insert(0, str(ROOT))
import bench  # noqa: E402


def _fake_smi(tmp_path: Path, lines) -> str:
    d = tmp_path / "bin"
    d.mkdir()
    exe = d / "nvidia-smi"
    body = "\n".join(f"echo '{l}'" for l in lines)
    exe.write_text(f"#!/bin/sh\n{body}\nexec sleep 30\n")
    exe.chmod(exe.stat().st_mode | stat.S_IEXEC)
    return str(d)


def test_clock_sampler_median_and_reasons(tmp_path, monkeypatch):
    rows = ["0, 2070, 2070, 950.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
            "0, 2055, 2070, 1210.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 1300.2, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
            "garbage line"]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, rows) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    s.start()
    time.sleep(0.5)
    r = s.stop()
    assert r["samples"] == 3 and r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_sampler_flags_thermal_slowdown(tmp_path, monkeypatch):
    rows = ["0, 1500, 2070, 1100.0, 0x40, Not Active, Active, Active, Not Active"]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, rows) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    s.start()
    time.sleep(0.5)
    r = s.stop()
    assert r["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"] and r["sm_mhz"] == 1500.0


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))  # nothing runnable there
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_traffic_is_reported_only_for_the_profiled_source(tmp_path, monkeypatch):
    assert bench.profiled_traffic() is not None  # the committed summary matches the source
    text = Path(bench.PROFILE_SUMMARY).read_text()
    stale = tmp_path / "stale.md"
    stale.write_text(text.replace(bench.kernel_source_hash(), "0" * 16))
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(stale))
    assert bench.profiled_traffic() is None
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(tmp_path / "missing.md"))
    assert bench.profiled_traffic() is None


def test_clock_sampler_leaves_idle_samples_out_of_the_median(tmp_path, monkeypatch):
    rows = ["0, 1980, 2070, 190.0, 0x0, Not Active, Not Active, Not Active, Not Active, 0",
            "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active, 97",
            "0, 2055, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Active, 100",
            "0, 1500, 2070, 200.0, 0x0, Not Active, Not Active, Not Active, Not Active, 3"]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, rows) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    s.start()
    time.sleep(0.5)
    r = s.stop()
    assert r["samples"] == 2 and r["samples_all"] == 4
    assert r["sm_mhz"] == (2070.0 + 2055.0) / 2
    assert r["reasons"] == ["sw_power_cap"]
