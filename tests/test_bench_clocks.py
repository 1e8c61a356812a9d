"""Host logic of bench.py: the clock record (a timed region shorter than the
sampling interval is still bracketed by samples, and the throttle reasons are
read from nvidia-smi's columns; nvidia-smi is faked by a script on PATH), and
the plan of graph replays that runs exactly K steps in input-set rotation."""
import os
import stat
import time

import bench


FAKE = """#!/bin/sh
i=0
while [ $i -lt 400 ]; do
  echo "0, 1965, 2070, 700.5, 0x4, Not Active, Not Active, Not Active, Active"
  sleep 0.05
  i=$((i+1))
done
"""


def _fake_smi(tmp_path, monkeypatch):
    f = tmp_path / "nvidia-smi"
    f.write_text(FAKE)
    f.chmod(f.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")


def test_short_region_is_bracketed(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch)
    clk = bench.ClockSampler(0)
    with clk:
        time.sleep(0.001)
    s = clk.summary()
    assert s["samples"] >= 2
    assert s["sm_mhz"] == 1965.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_long_region_keeps_the_samples_inside(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch)
    clk = bench.ClockSampler(0)
    with clk:
        time.sleep(0.5)
    assert clk.summary()["samples"] >= 6


def test_missing_tool_gives_an_empty_record(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    clk = bench.ClockSampler(0)
    with clk:
        pass
    assert clk.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_step_plan_runs_exactly_n_steps_in_set_rotation():
    # the timed region replays passes of `per` steps and then single steps;
    # expanded, step i must run on set i % nset and there must be n of them
    for nset in (1, 2, 3, 10):
        per = nset * max(1, bench.PASS_STEPS // nset)
        for n in (0, 1, 3, per - 1, per, per + 1, 2 * per + 7, 20000):
            passes, singles = bench.step_plan(n, nset, per)
            steps = [i % nset for i in range(per)] * passes + singles
            assert steps == [i % nset for i in range(n)]
