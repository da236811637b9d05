"""The bench's clock record (nvidia-smi samples taken during the timed region)
from synthetic sample lines: the median SM clock inside the window, the
largest maximum clock, and the throttle reasons that were active."""
import bench


def _line(sm, smax, power, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active"):
    return ["0", str(sm), str(smax), str(power), "0x0", hw, hw_th, sw_th, cap]


def _sampler(samples):
    s = bench.ClockSampler(0)
    s.samples = samples
    return s


def test_median_and_window():
    s = _sampler([(0.0, _line(900, 2070, 100)),             # before the window: ignored
                  (10.0, _line(2070, 2070, 300)), (10.2, _line(2040, 2070, 320)),
                  (10.4, _line(1980, 2070, 330)),
                  (20.0, _line(800, 2070, 90))])             # after it: ignored
    c = s.summary(10.0, 10.4)
    assert c["sm_mhz"] == 2040.0 and c["sm_max_mhz"] == 2070.0
    assert c["samples"] == 3 and c["reasons"] == [] and c["power_w_max"] == 330.0


def test_active_reasons_are_reported():
    s = _sampler([(1.0, _line(1800, 2070, 1400, cap="Active")),
                  (1.2, _line(1700, 2070, 1400, hw_th="Active", cap="Active"))])
    c = s.summary(1.0, 1.2)
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_no_samples_in_the_window_falls_back_to_all():
    s = _sampler([(5.0, _line(2070, 2070, 200))])
    assert s.summary(100.0, 101.0)["sm_mhz"] == 2070.0
    c = _sampler([]).summary(0.0, 1.0)
    assert c["samples"] == 0 and c["sm_mhz"] is None and c["reasons"] == ["no nvidia-smi samples"]


def test_unparsable_fields_are_skipped():
    s = _sampler([(1.0, _line("[N/A]", 2070, "[N/A]")), (1.1, _line(2000, "[N/A]", 250))])
    c = s.summary(1.0, 1.1)
    assert c["sm_mhz"] == 2000.0 and c["sm_max_mhz"] == 2070.0 and c["power_w_max"] == 250.0


def _nvml(samples, period=0.002):
    s = bench.NvmlClockSampler.__new__(bench.NvmlClockSampler)
    s.samples, s.period, s.which = samples, period, "index 0"
    return s


def test_nvml_samples_inside_a_short_region():
    # (time, SM MHz, max SM MHz, power W, clock-event reason bits)
    s = _nvml([(0.990, 1500.0, 2070.0, 150.0, 0x1),           # idle, before the region: ignored
               (1.000, 2070.0, 2070.0, 600.0, 0x0), (1.002, 2055.0, 2070.0, 620.0, 0x0),
               (1.004, 2070.0, 2070.0, 640.0, 0x4),            # power cap (kept, reported)
               (1.100, 900.0, 2070.0, 100.0, 0x0)])            # after: ignored
    c = s.summary(1.0, 1.005)
    assert c["samples"] == 3 and c["sm_mhz"] == 2070.0 and c["sm_mhz_min"] == 2055.0
    assert c["sm_max_mhz"] == 2070.0 and c["power_w_max"] == 640.0 and c["reasons"] == ["sw_power_cap"]


def test_nvml_throttle_bits_map_to_the_rejecting_reasons():
    s = _nvml([(5.0, 1200.0, 2070.0, 1400.0, 0x8 | 0x20 | 0x40)])
    assert s.summary(4.9, 5.1)["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_nvml_region_shorter_than_the_sampling_period():
    s = _nvml([(2.000, 2070.0, 2070.0, 500.0, 0), (2.040, 2040.0, 2070.0, 500.0, 0)])
    c = s.summary(2.010, 2.012)  # no sample inside: the nearest ones, and a note saying so
    assert c["samples"] == 2 and "nearest" in c["note"]
    c = _nvml([]).summary(0.0, 1.0)
    assert c["samples"] == 0 and c["sm_mhz"] is None
