"""bench.py's clock record on the CPU: the samples nvidia-smi writes during a
timed region (median SM clock under load, the throttle reasons seen), from
synthetic sample lines -- no GPU and no nvidia-smi needed."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

NOT = "Not Active"


def _line(sm, reasons=()):
    # index, clocks.sm, clocks.max.sm, power.draw, reasons.active, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap (the sampler's query order)
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ["Active" if n in reasons else NOT for n in names]
    return ", ".join(["0", str(sm), "2070", "900.5", "0x0"] + flags)


def _sampler(samples):
    c = bench.ClockSampler(0)
    c.lines = [(t, _line(sm, r)) for t, sm, r in samples]
    return c


def test_only_the_timed_region_counts():
    c = _sampler([(0.0, 900, ()), (1.00, 2070, ()), (1.02, 2070, ()), (1.04, 2040, ("sw_power_cap",)),
                  (1.06, 2070, ()), (2.0, 300, ("hw_slowdown",))])
    s = c.summary(1.0, 1.06)
    assert s["samples"] == 4
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]  # the idle samples outside the region carry no weight


def test_throttle_reasons_are_reported():
    c = _sampler([(1.0, 1500, ("hw_thermal_slowdown",)), (1.02, 1490, ("hw_slowdown", "sw_thermal_slowdown"))])
    s = c.summary(1.0, 1.02)
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1495.0


def test_no_samples_says_so():
    c = bench.ClockSampler(0)
    s = c.summary(0.0, 1.0)
    assert s["sm_mhz"] is None and s["reasons"] == ["no samples"]


def test_waiting_for_the_first_sample_is_bounded():
    c = bench.ClockSampler(0)  # never started: no process, returns at once
    c.wait_first(limit_s=0.5)
    assert c.lines == []
