"""The bench's clock record: nvidia-smi samples taken during the timed
region, read back as the median SM clock, the maximum and the throttle
reasons seen. Runs a stand-in nvidia-smi on PATH, so it needs no GPU."""

import os
import time

import bench

ROW = "0, {sm}, 2032, 812.5, 0x0, {hw}, Not Active, Not Active, {cap}"


def fake_smi(tmp_path, rows):
    """An executable named nvidia-smi that prints `rows` (then repeats the
    last one) every 20 ms until it is terminated; arguments are ignored."""
    script = tmp_path / "nvidia-smi"
    body = "".join(f"echo '{r}'\nsleep 0.02\n" for r in rows)
    script.write_text(f"#!/bin/sh\n{body}while true; do echo '{rows[-1]}'; sleep 0.02; done\n")
    script.chmod(0o755)
    return str(tmp_path)


def sample(monkeypatch, path, seconds=0.3):
    monkeypatch.setenv("PATH", path + os.pathsep + os.environ["PATH"])
    with bench.ClockSampler(0) as c:
        time.sleep(seconds)
    return c.summary()


def test_median_clock_and_power_cap(tmp_path, monkeypatch):
    rows = [ROW.format(sm=s, hw="Not Active", cap="Active") for s in (1900, 2032, 2032)]
    s = sample(monkeypatch, fake_smi(tmp_path, rows))
    assert s["samples"] >= 3
    assert s["sm_mhz"] == 2032.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"]


def test_hardware_slowdown_is_reported(tmp_path, monkeypatch):
    rows = [ROW.format(sm=1200, hw="Active", cap="Not Active")]
    s = sample(monkeypatch, fake_smi(tmp_path, rows))
    assert s["sm_mhz"] == 1200.0
    assert s["reasons"] == ["hw_slowdown"]


def test_no_samples_is_reported(tmp_path, monkeypatch):
    """A sampler that prints nothing usable leaves a reason, not silence."""
    s = sample(monkeypatch, fake_smi(tmp_path, ["garbage"]), seconds=0.1)
    assert s["sm_mhz"] is None and s["samples"] == 0
    assert s["reasons"] == ["no clock samples"]
