"""Host-side logic of bench.py that needs no GPU: the clock sampler's summary (only samples
inside the timed region count; NVML reason bits map to the throttle names the benchmark
reports) and its fallback when no clock source is available."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def sampler_with(samples, begin, end):
    c = bench.ClockSampler(0)
    c.nv = object()  # stands for an open NVML handle; summary() reads only the samples
    c.smax = 2032.0
    c.samples = samples
    c.t_begin, c.t_end = begin, end
    return c


def test_only_samples_inside_the_timed_region_count():
    c = sampler_with([(0.5, 900.0, 0x8), (1.0, 2000.0, 0), (1.5, 1900.0, 0), (2.0, 1800.0, 0),
                      (3.0, 500.0, 0x40)], 0.9, 2.1)
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1900.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == []  # the slowdown bits outside the region are not reported


def test_reason_bits_map_to_throttle_names():
    c = sampler_with([(1.0, 2000.0, 0x4), (1.1, 1990.0, 0x8 | 0x20), (1.2, 1980.0, 0x40)], 0.0, 9.0)
    assert c.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap",
                                      "sw_thermal_slowdown"]


def test_no_clock_source_is_reported_not_invented():
    c = bench.ClockSampler(0)  # neither NVML nor nvidia-smi was started
    s = c.summary()
    assert s["sm_mhz"] is None and s["reasons"] == ["clock sampling unavailable"]
