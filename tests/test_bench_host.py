"""Host-side logic of bench.py that needs no GPU (CPU only).

The clock sampler reads nvidia-smi's CSV stream in a background thread; the
bench keeps only the samples of its timed region and flags a run whose clocks
were throttled.  A fake nvidia-smi on PATH stands in for the tool.
"""
import os
import stat
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def fake_smi(tmp_path, lines, period_s=0.02):
    """An nvidia-smi that prints the given CSV lines in a loop (the last one repeated)."""
    script = tmp_path / "nvidia-smi"
    body = "\n".join(f'echo "{ln}"; sleep {period_s}' for ln in lines)
    last = lines[-1]
    script.write_text(f"#!/bin/bash\n{body}\nwhile true; do echo \"{last}\"; sleep {period_s}; done\n")
    script.chmod(script.stat().st_mode | stat.S_IEXEC)
    return str(tmp_path)


@pytest.fixture
def bench_mod():
    import bench
    return bench


def row(sm, smax=2070, reasons=("Not Active",) * 4):
    return ", ".join(["0", str(sm), str(smax), "900.0", "0x0"] + list(reasons))


def test_sampler_keeps_the_timed_window(bench_mod, monkeypatch, tmp_path):
    # 5 idle samples at 1000 MHz, then the loaded clock; the window excludes the idle ones
    path = fake_smi(tmp_path, [row(1000)] * 5 + [row(2070)])
    monkeypatch.setenv("PATH", path + os.pathsep + os.environ["PATH"])
    s = bench_mod.ClockSampler(0)
    s.wait()
    time.sleep(0.3)
    start = s.mark()
    time.sleep(0.2)
    end = s.mark()
    out = s.stop(start, end)
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == [] and out["samples"] >= 3


def test_sampler_reports_throttle_reasons(bench_mod, monkeypatch, tmp_path):
    hot = ("Not Active", "Not Active", "Active", "Not Active")  # sw_thermal_slowdown
    path = fake_smi(tmp_path, [row(1800, reasons=hot)])
    monkeypatch.setenv("PATH", path + os.pathsep + os.environ["PATH"])
    s = bench_mod.ClockSampler(0)
    s.wait()
    start = s.mark()
    time.sleep(0.1)
    out = s.stop(start, s.mark())
    assert out["reasons"] == ["sw_thermal_slowdown"] and out["sm_mhz"] == 1800.0


def test_sampler_without_nvidia_smi(bench_mod, monkeypatch, tmp_path):
    monkeypatch.setenv("PATH", str(tmp_path))  # no nvidia-smi anywhere
    s = bench_mod.ClockSampler(0)
    s.wait(0.1)
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_roofline_peak_follows_the_power_cap(bench_mod):
    peaks = {"bf16_burst": 1926.9, "bf16_sustained": 1715.2}
    assert bench_mod.roofline_peak(peaks, {"reasons": []}) == (1926.9, "burst")
    assert bench_mod.roofline_peak(peaks, {"reasons": ["sw_power_cap"]}) == (1715.2, "sustained")
