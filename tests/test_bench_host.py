"""Host-side pieces of bench.py: clock-sample filtering and the traffic record's guard."""
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


def test_traffic_is_reported_only_for_the_sources_it_was_captured_with(monkeypatch):
    now = bench.sources_sha256()
    monkeypatch.setitem(bench.TRAFFIC, "sources_sha256", now)
    assert bench.recorded_traffic(True, 1) == bench.TRAFFIC["bytes_per_launch"]
    assert bench.recorded_traffic(False, 1) is None and bench.recorded_traffic(True, 2) is None
    monkeypatch.setitem(bench.TRAFFIC, "sources_sha256", "0" * 64)
    assert bench.recorded_traffic(True, 1) is None


def test_var_rank_grid_keeps_the_large_products_tiles():
    import numpy as np
    import tlr_inputs as ti
    p = ti.var_rank_grid(4096)
    assert p.A.b == 1024 and p.m == p.n == 4096 and p.budget == (2 << 30) // 64
    r = np.asarray(p.A.ranks).reshape(4, 4)
    for i in range(4):
        for j in range(4):
            if i != j:
                want = min(256, max(8, int(np.floor(256 * np.exp(-abs(i - j) / 4.0) + 0.5))))
                assert r[i, j] == want
