"""Host-side logic of the benchmark that needs no GPU: the clock record taken
during the timed region (median SM clock, the throttle reasons seen, the
fallback for a region shorter than the sampling period)."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _sampler(rows):
    """A ClockSampler holding the given (time, fields) samples, without
    starting nvidia-smi."""
    s = object.__new__(bench.ClockSampler)
    s.samples = [(t, [x.strip() for x in line.split(",")]) for t, line in rows]
    s.proc = None
    return s


NA, A = "Not Active", "Active"


def row(sm, power, hw=NA, hwt=NA, swt=NA, cap=NA):
    return "%s, 2070, %s, %s, %s, %s, %s" % (sm, power, hw, hwt, swt, cap)


def test_median_clock_and_reasons_inside_the_window_only():
    s = _sampler([(0.5, row(1200, 100, hw=A)),          # before the window
                  (1.0, row(2070, 300)), (1.1, row(2070, 350, cap=A)),
                  (1.2, row(2050, 320)), (1.3, row(2070, 310)),
                  (2.5, row(900, 90, hwt=A))])          # after it
    c = s.summary(1.0, 2.0)
    assert c["samples"] == 4 and c["note"] == "inside timed region"
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]             # kept and noted, not a rejection
    assert c["power_w_max"] == 350


def test_every_slowdown_reason_is_reported():
    s = _sampler([(1.0, row(1500, 200, hw=A)), (1.1, row(1500, 200, hwt=A)),
                  (1.2, row(1500, 200, swt=A))])
    assert s.summary(0.9, 1.3)["reasons"] == ["hw_slowdown", "hw_thermal_slowdown",
                                              "sw_thermal_slowdown"]


def test_short_region_takes_the_nearest_samples_after_it_started():
    s = _sampler([(0.9, row(2070, 100)), (1.25, row(2060, 300)), (1.35, row(2070, 310)),
                  (1.45, row(2070, 320)), (1.55, row(2070, 330))])
    c = s.summary(1.2, 1.21)
    assert c["samples"] == 3 and c["note"].startswith("timed region shorter")
    assert c["sm_mhz"] == 2070


def test_no_samples_gives_an_empty_record():
    c = _sampler([]).summary(0.0, 1.0)
    assert c == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_unparsable_fields_are_skipped():
    s = _sampler([(1.0, "[N/A], 2070, [N/A], Not Active, Not Active, Not Active, Not Active"),
                  (1.1, row(2070, 250))])
    c = s.summary(0.9, 1.2)
    assert c["sm_mhz"] == 2070 and c["power_w_max"] == 250 and c["reasons"] == []
