"""Host-side pieces of bench.py: clock-sample filtering and the traffic record's hash."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_clock_summary_keeps_samples_inside_the_timed_region():
    c = bench.ClockSampler(0)
    row = lambda mhz, cap: ["0", str(mhz), "2070", "900", "0x0", "Not Active", "Not Active", "Not Active", cap]
    c.samples = [row(1200, "Not Active"), row(2070, "Active"), row(2055, "Active"), row(900, "Not Active")]
    c.times = [1.0, 2.0, 2.5, 4.0]
    c.t0, c.t1 = 1.5, 3.0
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] in (2055.0, 2070.0) and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_throttle_reasons_and_no_samples():
    c = bench.ClockSampler(0)
    assert c.summary()["reasons"] == ["no samples"]
    c.samples = [["0", "1500", "2070", "1000", "0x8", "Active", "Not Active", "Active", "Not Active"]]
    c.times = [1.0]
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_traffic_record_matches_the_kernel_sources():
    # the DRAM bytes in bench.py were captured with these sources; a kernel change
    # must come with a new capture (or the bench reports null traffic)
    assert bench.sources_sha256() == bench.TRAFFIC["sources_sha256"]
