"""The bench's clock record: samples are taken only while the timed regions (and, for regions shorter than the
sampling interval, untimed replays of the same work) run, throttle reasons are parsed, and a missing nvidia-smi
gives no record instead of an error.  A fake nvidia-smi on PATH stands in for the real one (no GPU needed)."""
import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def fake_smi(tmp_path, line):
    exe = tmp_path / "nvidia-smi"
    exe.write_text("#!/bin/sh\nwhile true; do echo '%s'; sleep 0.03; done\n" % line)
    exe.chmod(exe.stat().st_mode | stat.S_IEXEC)
    return str(tmp_path)


def test_short_region_is_held_until_sampled(tmp_path, monkeypatch):
    line = "1965, 2070, 812.50, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
    monkeypatch.setenv("PATH", fake_smi(tmp_path, line) + os.pathsep + os.environ["PATH"])
    calls = []
    with bench.ClockSampler(0) as clk:
        assert clk.stamped, "the sampler is running before the timed region starts"
        time.sleep(0.002)                       # a timed region of a few milliseconds
        clk.hold(lambda: (calls.append(1), time.sleep(0.01)))
    s = clk.summary()
    assert calls, "short regions are extended with untimed replays"
    assert s["window_s"] >= bench.ClockSampler.MIN_WINDOW_S
    assert s["samples"] >= 3
    assert s["sm_mhz"] == 1965.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_long_region_needs_no_replay(tmp_path, monkeypatch):
    line = "2070, 2070, 900.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
    monkeypatch.setenv("PATH", fake_smi(tmp_path, line) + os.pathsep + os.environ["PATH"])
    calls = []
    with bench.ClockSampler(0) as clk:
        time.sleep(bench.ClockSampler.MIN_WINDOW_S + 0.05)
        clk.hold(lambda: calls.append(1))
    s = clk.summary()
    assert not calls
    assert s["reasons"] == [] and s["sm_mhz"] == 2070.0


def test_no_nvidia_smi_gives_no_record(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    with bench.ClockSampler(0) as clk:
        clk.hold(lambda: (_ for _ in ()).throw(AssertionError("no replay without a sampler")))
    assert clk.summary() is None
