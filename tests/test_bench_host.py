"""Host logic of bench.py (no GPU): which FP8 denominator a roofline takes, and the
clock-record summary it is chosen from."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_fp8_peak_sustained_only_under_the_power_cap():
    b = _bench()
    burst, sustained = 1805.2, 1405.8
    peak, src = b._fp8_peak(burst, sustained, "measured", {"reasons": ["sw_power_cap"]})
    assert peak == 2 * sustained and "sustained" in src
    peak, src = b._fp8_peak(burst, sustained, "measured", {"reasons": []})
    assert peak == 2 * burst and "burst" in src
    # a clock record without samples, or no sustained figure: the burst figure
    assert b._fp8_peak(burst, sustained, "measured", {})[0] == 2 * burst
    assert b._fp8_peak(burst, None, "measured", {"reasons": ["sw_power_cap"]})[0] == 2 * burst


def test_clock_summary_reads_reasons_and_median():
    b = _bench()
    s = b.ClockSampler(0)
    # index, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    s.lines = [
        "0, 1800, 2032, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2032, 2032, 500.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1900, 2032, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
    ]
    out = s.summary()
    assert out["sm_mhz"] == 1900 and out["sm_max_mhz"] == 2032 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
