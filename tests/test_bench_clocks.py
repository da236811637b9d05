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
