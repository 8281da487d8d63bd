"""Host logic of bench.py that needs no GPU: the clock record keeps the
samples of the timed region only and names their clock-event reasons."""

import os
import sys
import threading

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sampler(samples, max_mhz=2070):
    """An NVML sampler holding given samples (no NVML: its thread has ended)."""
    s = object.__new__(bench.NvmlSampler)
    s.samples = list(samples)
    s.max_mhz = max_mhz
    s.stop_ev = threading.Event()
    s.th = threading.Thread(target=lambda: None)
    s.th.start()
    return s


def test_clock_record_keeps_the_timed_region():
    # idle before (GPU idle bit), two samples inside (one under the power cap),
    # a slowdown after the region: only the two inside count
    s = _sampler([(0.0, 1000, 0x1), (1.0, 2070, 0x0), (1.5, 2060, 0x4), (3.0, 900, 0x8)])
    r = s.stop(0.5, 2.0)
    assert r["samples"] == 2
    assert r["sm_mhz"] == 2065
    assert r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_record_names_every_rejecting_reason():
    s = _sampler([(1.0, 1500, 0x8 | 0x20 | 0x40), (1.1, 1600, 0x80)])
    r = s.stop(0.0, 2.0)
    assert r["reasons"] == ["hw_power_brake_slowdown", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_record_without_samples_inside_says_so():
    s = _sampler([(0.0, 2070, 0x0), (5.0, 2070, 0x0)])
    r = s.stop(1.0, 2.0)
    assert r["samples"] == 0 and "none inside" in r["source"]
    assert _sampler([]).stop(0.0, 1.0) is None
