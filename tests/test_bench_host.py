"""Host-side pieces of bench.py that need no GPU: the clock sampler that runs during the
timed region, driven here by a stand-in ``nvidia-smi`` on PATH that prints the same CSV
columns, and the rule that only samples taken after the timed region starts count."""
import os
import stat
import time

import bench

_FAKE_SMI = r"""#!/usr/bin/env python3
# Stand-in for nvidia-smi --query-gpu=... --format=csv,noheader,nounits -lms 200:
# one warm-up sample with a hardware slowdown, then, once the go-file exists, timed
# samples at 1965/2070 MHz with the power cap active.
import os, sys, time
go = os.environ["FAKE_SMI_GO"]
print("0, 1200, 2070, 900.0, 0x8, Active, Not Active, Not Active, Not Active", flush=True)
while not os.path.exists(go):
    time.sleep(0.02)
for mhz in (1965, 1950, 1980, 1965, 1965):
    print(f"0, {mhz}, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
          flush=True)
    time.sleep(0.02)
time.sleep(60)
"""


def _install_fake(tmp_path, monkeypatch):
    smi = tmp_path / "bin" / "nvidia-smi"
    smi.parent.mkdir()
    smi.write_text(_FAKE_SMI)
    smi.chmod(smi.stat().st_mode | stat.S_IXUSR)
    monkeypatch.setenv("PATH", str(smi.parent) + os.pathsep + os.environ["PATH"])
    go = tmp_path / "go"
    monkeypatch.setenv("FAKE_SMI_GO", str(go))
    return go


def test_clock_sampler_counts_only_the_timed_region(tmp_path, monkeypatch):
    go = _install_fake(tmp_path, monkeypatch)
    clk = bench.ClockSampler(0, str(tmp_path / "out" / "clocks_gpu{gpu}.csv"))
    clk.start()
    clk.mark()                       # the warm-up sample is before this point
    go.touch()
    deadline = time.time() + 20
    while time.time() < deadline:
        if sum(1 for _ in open(clk.path)) >= 6:
            break
        time.sleep(0.05)
    rec = clk.stop()
    assert clk.path.endswith(os.path.join("out", "clocks_gpu0.csv"))
    assert rec["samples"] == 5
    assert rec["sm_mhz"] == 1965.0
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"]      # the warm-up hw_slowdown is not counted


def test_clock_sampler_without_nvidia_smi_reports_unsampled(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))      # no nvidia-smi anywhere
    clk = bench.ClockSampler(3)
    assert os.path.basename(clk.path) == "mok_bench_clocks_gpu3.csv"
    clk.start()
    clk.mark()
    assert clk.stop() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
