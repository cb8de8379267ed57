"""Host logic of bench.py's clock record, on the CPU: the summary of the NVML readings (median SM
clock, the clock-event reasons seen in any reading, the sample count) and the bits it decodes.
The readings themselves need a GPU and its driver; here they are given.
"""
import bench


def _sampler(samples, max_mhz=2032):
    s = object.__new__(bench.ClockSampler)  # no NVML: the readings are set by hand
    s.ok, s.err, s.samples, s.max_mhz = True, "", list(samples), max_mhz
    return s


def test_summary_median_and_reasons():
    s = _sampler([(2032, 0x0), (1965, 0x4), (2032, 0x1)])
    out = s.summary()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2032  # median of 1965, 2032, 2032
    assert out["sm_max_mhz"] == 2032
    # sw_power_cap is reported; gpu_idle is not a reason for the record
    assert out["reasons"] == ["sw_power_cap"]


def test_summary_reports_slowdowns():
    s = _sampler([(1500, 0x8 | 0x40), (1600, 0x20)])
    assert set(s.summary()["reasons"]) == {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def test_summary_without_samples_or_nvml():
    assert _sampler([]).summary() == {"sm_mhz": None, "sm_max_mhz": 2032, "reasons": [], "samples": 0}
    s = _sampler([])
    s.ok, s.err = False, "OSError('libnvidia-ml.so.1')"
    out = s.summary()
    assert out["sm_mhz"] is None and "NVML unavailable" in out["note"]


def test_sample_appends_reading_from_nvml():
    class FakeNvml:
        def sm(self):
            return 1980

        def reasons(self):
            return 0x4

    s = _sampler([])
    s.nv = FakeNvml()
    s.sample()
    s.sample()
    assert s.samples == [(1980, 0x4), (1980, 0x4)]
    assert s.summary()["sm_mhz"] == 1980
