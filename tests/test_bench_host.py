"""Host-side logic of the benchmark that needs no GPU: the clock record taken
during the timed region (median SM clock, the throttle reasons seen, samples
only from inside the window), the sampling thread's start / stop order with a
fake reader in place of NVML, and the nvidia-smi fallback's line parser."""
import os
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def smp(t, sm, power, *reasons, smax=2070.0):
    return (t, float(sm), smax, float(power), frozenset(reasons))


def test_median_clock_and_reasons_inside_the_window_only():
    s = bench.ClockSampler.from_samples([
        smp(0.5, 1200, 100, "hw_slowdown"),                 # before the window
        smp(1.0, 2070, 300), smp(1.1, 2070, 350, "sw_power_cap"),
        smp(1.2, 2050, 320), smp(1.3, 2070, 310),
        smp(2.5, 900, 90, "hw_thermal_slowdown")])          # after it
    c = s.summary(1.0, 2.0)
    assert c["samples"] == 4 and c["note"] == "inside timed region"
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]             # kept and noted, not a rejection
    assert c["power_w_max"] == 350
    assert s.count(1.0, 2.0) == 4 and s.count(0.0, 0.9) == 1


def test_every_slowdown_reason_is_reported():
    s = bench.ClockSampler.from_samples([smp(1.0, 1500, 200, "hw_slowdown"),
                                         smp(1.1, 1500, 200, "hw_thermal_slowdown"),
                                         smp(1.2, 1500, 200, "sw_thermal_slowdown")])
    assert s.summary(0.9, 1.3)["reasons"] == ["hw_slowdown", "hw_thermal_slowdown",
                                              "sw_thermal_slowdown"]


def test_no_samples_gives_an_empty_record():
    c = bench.ClockSampler.from_samples([]).summary(0.0, 1.0)
    assert c == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_missing_fields_are_skipped():
    s = bench.ClockSampler.from_samples([(1.0, None, 2070.0, None, frozenset()),
                                         smp(1.1, 2070, 250)])
    c = s.summary(0.9, 1.2)
    assert c["sm_mhz"] == 2070 and c["power_w_max"] == 250 and c["reasons"] == []


def test_sampling_thread_covers_a_few_millisecond_region():
    """The benchmark's order: start the sampler, run the timed region, stop,
    then summarise.  A 1 ms period leaves several samples inside a region of a
    few milliseconds (the 20-step region is about 5 ms)."""
    calls = []

    def reader():
        calls.append(time.time())
        return 2070.0, 2070.0, 400.0, frozenset()
    s = bench.ClockSampler(reader=reader, period_s=0.001)
    time.sleep(0.01)
    t0 = time.time()
    time.sleep(0.006)                                    # the "timed region"
    t1 = time.time()
    time.sleep(0.005)
    s.stop()
    n_after_stop = len(s.samples)
    time.sleep(0.005)
    assert len(s.samples) == n_after_stop                # stopped means stopped
    c = s.summary(t0, t1)
    assert c["samples"] >= 2 and c["sm_mhz"] == 2070 and c["source"].startswith("nvml")


def test_reader_failures_are_not_samples():
    s = bench.ClockSampler(reader=lambda: None, period_s=0.001)
    time.sleep(0.005)
    s.stop()
    assert s.samples == []


def test_nvidia_smi_line_parser():
    line = "2070, 2070, 310.5, Not Active, Not Active, Not Active, Active"
    assert bench.ClockSampler.parse_smi(line) == (2070.0, 2070.0, 310.5,
                                                  frozenset({"sw_power_cap"}))
    sm, smax, power, reasons = bench.ClockSampler.parse_smi(
        "[N/A], 2070, [N/A], Active, Not Active, Active, Not Active")
    assert sm is None and power is None and reasons == {"hw_slowdown", "sw_thermal_slowdown"}
    assert bench.ClockSampler.parse_smi("2070, 2070") is None
