"""Host logic of the bench's clock record: the decoding of NVML clock-event
reason bits and the median over loaded samples (no GPU, no NVML)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _sampler(samples, sm_max):
    sys.path.insert(0, ROOT)
    import bench
    c = object.__new__(bench.ClockSampler)
    c.nvml, c.proc = object(), None
    c.samples, c.sm_max = samples, sm_max
    return c


def test_reason_bits_decode():
    # 0x1 (idle) and 0x10 (sync boost) are not reported; 0x4 | 0x40 are
    s = _sampler([(2070.0, 0x1), (2070.0, 0x4 | 0x10), (1900.0, 0x40)], 2070.0).summary()
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert s["samples"] == 3 and s["sm_max_mhz"] == 2070.0


def test_median_ignores_idle_samples():
    # samples below half the maximum clock are idle gaps, not load
    s = _sampler([(345.0, 0), (2070.0, 0), (2055.0, 0), (2070.0, 0)], 2070.0).summary()
    assert s["sm_mhz"] == 2070.0 and s["reasons"] == []


def test_all_idle_keeps_every_sample():
    s = _sampler([(300.0, 0), (400.0, 0)], 2070.0).summary()
    assert s["sm_mhz"] == 350.0
