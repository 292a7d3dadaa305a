"""The clock record of the bench line (CPU only, with a stand-in for nvidia-smi).

bench.py samples SM clocks and throttle reasons with nvidia-smi during the timed
region; a run whose record shows a hardware or thermal slowdown is rejected, and
one stuck below its maximum clock with no reason is suspect.  This checks the
parsing: the median is taken over the samples under load (idle samples at the
edges of the region left out), malformed lines are skipped, and every reason
seen active in any sample is reported.
"""
import os
import stat

import bench

SAMPLES = [
    "0, 345, 2070, 120.50, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "0, 2070, 2070, 1210.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "[N/A], [N/A]",
    "0, 2055, 2070, 1392.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
    "0, 2070, 2070, 1300.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
]


def fake_smi(tmp_path, lines):
    script = tmp_path / "nvidia-smi"
    body = "\n".join(f"echo '{line}'" for line in lines)
    script.write_text(f"#!/bin/sh\n{body}\nexec sleep 30\n")
    script.chmod(script.stat().st_mode | stat.S_IEXEC)
    return str(tmp_path)


def test_clock_record_from_samples(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", fake_smi(tmp_path, SAMPLES) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    s.start()
    rec = s.stop()
    assert rec["samples"] == 4                      # the malformed line is skipped
    assert rec["sm_mhz"] == 2070.0                  # median of 2070, 2055, 2070 (the 345 MHz idle sample left out)
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"]       # any sample with the reason active reports it


def test_hardware_slowdown_is_reported(tmp_path, monkeypatch):
    lines = ["0, 1500, 2070, 1000.0, 0x8, Active, Not Active, Not Active, Not Active",
             "0, 1400, 2070, 1000.0, 0x28, Active, Active, Not Active, Not Active"]
    monkeypatch.setenv("PATH", fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    s.start()
    rec = s.stop()
    assert rec["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert rec["sm_mhz"] == 1450.0


def test_missing_nvidia_smi_is_stated(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))  # an empty directory: no nvidia-smi
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]
