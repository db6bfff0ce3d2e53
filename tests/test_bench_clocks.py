"""bench.py's clock record, on the host: samples in nvidia-smi's CSV format are
filtered to the timed window and summarised (median SM clock, maximum, throttle
reasons that were active, power); with a window shorter than the sampling
interval the nearest sample is used."""
import os
import time

import pytest

import bench


class _Done:
    """Stands in for the nvidia-smi process that has been sampling."""

    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _stamp(t):
    lt = time.localtime(t)
    return time.strftime("%Y/%m/%d %H:%M:%S", lt) + ".%03d" % int(round((t % 1) * 1000) % 1000)


def _row(t, sm, power=400.0, hw="Not Active", thermal="Not Active", sw_thermal="Not Active", cap="Not Active"):
    return f"{_stamp(t)}, {sm}, 2070, {power}, 0x0, {hw}, {thermal}, {sw_thermal}, {cap}"


def _sampler(rows, window):
    s = bench.ClockSampler(0)
    s.out.write("\n".join(rows) + "\n")
    s.out.flush()
    s.proc = _Done()
    if window is not None:
        s.mark(*window)
    return s


@pytest.fixture(autouse=True)
def _no_sleep(monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda _s: None)


def test_window_filters_and_summarises():
    t0 = 1_780_000_000.0
    rows = [_row(t0 - 1.0, 1200.0, power=150.0),                     # before the window
            _row(t0 + 0.10, 2055.0, power=480.0, cap="Active"),
            _row(t0 + 0.15, 2070.0, power=470.0),
            _row(t0 + 0.20, 2040.0, power=490.0),
            _row(t0 + 2.0, 900.0, power=100.0, thermal="Active")]     # after it
    out = _sampler(rows, (t0, t0 + 0.5)).stop()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]            # the thermal sample lies outside
    assert out["power_w_max"] == 490.0


def test_short_window_takes_the_nearest_sample():
    t0 = 1_780_000_000.0
    rows = [_row(t0, 2000.0), _row(t0 + 0.05, 2060.0, hw="Active"), _row(t0 + 0.10, 1990.0)]
    out = _sampler(rows, (t0 + 0.051, t0 + 0.052)).stop()
    assert out["samples"] == 1 and out["sm_mhz"] == 2060.0
    assert out["reasons"] == ["hw_slowdown"]


def test_no_samples_and_no_tool():
    assert _sampler([], None).stop()["reasons"] == ["no samples"]
    s = bench.ClockSampler(0)
    s.proc = None
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]
    os.unlink(s.out.name)
