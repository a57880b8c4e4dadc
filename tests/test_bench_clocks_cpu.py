"""The benchmark's clock record: the median SM clock under load, the maximum
clock, the peak and mean power and the throttle reasons active during the timed
region, read from nvidia-smi's CSV samples.  A fake nvidia-smi on PATH
stands in for the tool, so this runs without a GPU."""
import os
import stat
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

SAMPLES = [
    "1400, 2070, 1398.50, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
    "1500, 2070, 1201.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "[N/A], 2070, [N/A], 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "1450, 2070, 1300.25, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
    "garbled line",
]


def _fake_smi(tmp_path, lines):
    path = tmp_path / "nvidia-smi"
    body = "".join(f"echo '{ln}'\n" for ln in lines)
    path.write_text("#!/bin/sh\n" + body + "exec sleep 30\n")
    path.chmod(path.stat().st_mode | stat.S_IXUSR)
    return str(tmp_path)


def _sample(monkeypatch, tmp_path, lines):
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, lines) + os.pathsep + os.environ.get("PATH", ""))
    with bench.ClockSampler(0) as clk:
        pass
    return clk.summary()


def test_summary_of_samples(monkeypatch, tmp_path):
    s = _sample(monkeypatch, tmp_path, SAMPLES)
    assert s["samples"] == 4  # the garbled line is dropped
    assert s["sm_mhz"] == 1450.0  # median of 1400, 1500, 1450; [N/A] is skipped
    assert s["sm_max_mhz"] == 2070.0
    assert s["power_w_max"] == 1398.5
    assert abs(s["power_w_mean"] - (1398.5 + 1201.0 + 1300.25) / 3) < 1e-9  # the energy per step uses the mean
    assert s["reasons"] == ["sw_power_cap"]


def test_slowdown_reasons_are_reported(monkeypatch, tmp_path):
    lines = ["1200, 2070, 900.0, 0x0000000000000008, Active, Not Active, Active, Not Active"]
    s = _sample(monkeypatch, tmp_path, lines)
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_no_tool_means_unsampled(monkeypatch, tmp_path):
    monkeypatch.setenv("PATH", str(tmp_path))  # an empty directory: no nvidia-smi
    with bench.ClockSampler(0) as clk:
        pass
    assert clk.summary()["reasons"] == ["unsampled"]
