"""bench.py's clock sampler against a stand-in nvidia-smi (CPU only).

The sampler drops the first sample (taken before the timed region), reports
the median SM clock, the maximum clock and power seen and every throttle
reason that was active in any sample; without nvidia-smi it says so instead
of failing.
"""
import os
import stat
import sys

import pytest


def _fake_smi(tmp_path, lines):
    """A stand-in that prints one sample every 50 ms, as `nvidia-smi -lms 50` does."""
    script = tmp_path / "nvidia-smi"
    body = "\nsleep 0.05\n".join(f"echo '{ln}'" for ln in lines)
    script.write_text("#!/bin/sh\n" + body + "\nwhile true; do sleep 0.05; done\n")
    script.chmod(script.stat().st_mode | stat.S_IXUSR)
    return str(tmp_path)


@pytest.fixture
def bench_mod():
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    return bench


def test_clock_sampler_reports_median_clock_and_active_reasons(tmp_path, monkeypatch, bench_mod):
    lines = [
        "0, 1500, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # before timing: dropped
        "0, 2070, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2040, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    c = bench_mod.Clocks(0)
    c.start()
    import time
    time.sleep(0.5)
    r = c.stop()
    assert r["samples"] == 3
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["power_w_max"] == 1000.0
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_sampler_flags_thermal_slowdown(tmp_path, monkeypatch, bench_mod):
    lines = [
        "0, 2070, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1200, 2070, 900.0, 0x40, Not Active, Active, Not Active, Not Active",
    ]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    c = bench_mod.Clocks(0)
    c.start()
    import time
    time.sleep(0.4)
    r = c.stop()
    assert r["reasons"] == ["hw_thermal_slowdown"] and r["sm_mhz"] == 1200.0


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch, bench_mod):
    monkeypatch.setenv("PATH", str(tmp_path))     # an empty directory: no nvidia-smi
    c = bench_mod.Clocks(0)
    c.start()
    r = c.stop()
    assert r["sm_mhz"] is None and r["reasons"] == ["nvidia-smi unavailable"]
