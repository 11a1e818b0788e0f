"""The bench's choice of the bf16 peak a timed region is compared with
(CPU only): burst unless a long region ran under the power cap at a lower
clock."""

import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PEAKS = {"bf16_tflops": 1976.9, "bf16_tflops_sustained": 1752.8}


def bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def clocks(reasons, sm, smax=2070.0):
    return {"reasons": reasons, "sm_mhz": sm, "sm_max_mhz": smax, "samples": 100}


def test_short_region_takes_the_burst_peak_even_under_the_cap():
    peak, kind, _ = bench().choose_peak(PEAKS, clocks(["sw_power_cap"], 1800.0), 0.2)
    assert (peak, kind) == (1976.9, "burst")


def test_long_region_without_the_cap_takes_the_burst_peak():
    peak, kind, _ = bench().choose_peak(PEAKS, clocks([], 2070.0), 5.0)
    assert (peak, kind) == (1976.9, "burst")


def test_cap_that_held_the_clock_keeps_the_burst_peak():
    peak, kind, why = bench().choose_peak(PEAKS, clocks(["sw_power_cap"], 2070.0), 1.7)
    assert (peak, kind) == (1976.9, "burst") and "clock held" in why


def test_long_capped_and_slowed_region_takes_the_sustained_peak():
    peak, kind, _ = bench().choose_peak(PEAKS, clocks(["sw_power_cap"], 1900.0), 1.7)
    assert (peak, kind) == (1752.8, "sustained")
