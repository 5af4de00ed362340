"""CPU checks of the bench line's clock record: nvidia-smi rows are parsed,
only the samples inside the timed region count when there are any, and the
throttle reasons that reject a run (hw_slowdown, hw_thermal_slowdown,
sw_thermal_slowdown) or are noted (sw_power_cap) come through by name."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def row(mhz, power_cap="Not Active", hw="Not Active", thermal="Not Active"):
    # index, clocks.sm, clocks.max.sm, power.draw, reasons.active, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return f"0, {mhz}, 2070, 1100.5, 0x0, {hw}, Not Active, {thermal}, {power_cap}"


def sampler(rows, t0=None, t1=None):
    c = bench.ClockSampler(0)
    c.rows = list(rows)
    c.t0, c.t1 = t0, t1
    return c


def test_inside_the_timed_region_only():
    c = sampler([(1.0, row(1500)), (2.0, row(2070)), (2.5, row(2060)), (3.0, row(2070)), (9.0, row(900))],
                t0=1.9, t1=3.1)
    s = c.summary()
    assert s["in_timed_region"] and s["samples"] == 3
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["reasons"] == []


def test_reasons_by_name():
    c = sampler([(1.0, row(1950, power_cap="Active")), (1.1, row(1800, hw="Active", thermal="Active"))],
                t0=0.5, t1=2.0)
    s = c.summary()
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1875


def test_outside_samples_when_none_inside_and_garbage_skipped():
    c = sampler([(1.0, row(2000)), (1.2, "[Not Supported]"), (1.4, row(2040))], t0=5.0, t1=6.0)
    s = c.summary()
    assert not s["in_timed_region"] and s["samples"] == 2 and s["sm_mhz"] == 2020


def test_no_samples():
    s = sampler([]).summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == ["unavailable"]
