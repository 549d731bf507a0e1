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
    assert bench.recorded_traffic(True, 1, True) == bench.TRAFFIC["bytes_per_launch"]
    assert bench.recorded_traffic(False, 1, True) is None and bench.recorded_traffic(True, 2, True) is None
    assert bench.recorded_traffic(True, 1, False) is None      # captured on the per-triple plan only
    monkeypatch.setitem(bench.TRAFFIC, "sources_sha256", "0" * 64)
    assert bench.recorded_traffic(True, 1, True) is None


def test_recorded_traffic_matches_the_current_kernel_sources():
    assert bench.TRAFFIC["sources_sha256"] == bench.sources_sha256()


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


def test_peak_follows_the_length_of_the_timed_region():
    """Burst peak for a region shorter than three seconds, sustained from three on;
    fp32 products are compared with the tf32 peak (bf16 x 1.1 / 2.25)."""
    assert bench.peak_choice(74.0) == "burst" and bench.peak_choice(2999.0) == "burst"
    assert bench.peak_choice(3000.0) == "sustained"
    peaks = {"bf16_tflops": 1878.3, "bf16_tflops_sustained": 1704.2, "hbm_gbs": 6784.5}
    assert bench.dtype_peaks("bf16", peaks) == (1878.3, 1704.2)
    b, s = bench.dtype_peaks("f32", peaks)
    assert abs(b - 1878.3 * 1.1 / 2.25) < 1e-9 and abs(s - 1704.2 * 1.1 / 2.25) < 1e-9


def test_algorithmic_bytes_count_inputs_once_and_c_once_or_twice():
    import tlr_inputs as ti
    p = ti.problem(2, scale_down=4)                     # beta != 0: C read and written
    assert bench.algorithmic_bytes(p) == bench.input_bytes(p) + 2 * p.m * p.n * 4
    q = ti.problem(1)                                   # beta == 0: C written only
    assert bench.algorithmic_bytes(q) == bench.input_bytes(q) + q.m * q.n * 4
    assert bench.input_bytes(q) == q.A.nbytes_device() + q.B.nbytes_device()


def test_near_gpu_restores_the_affinity(monkeypatch):
    before = os.sched_getaffinity(0)
    monkeypatch.setattr(bench, "gpu_local_cpus", lambda i: sorted(before)[:1])
    with bench.near_gpu(0) as n:
        assert os.sched_getaffinity(0) == set(sorted(before)[:1]) and n.cpus == sorted(before)[:1]
    assert os.sched_getaffinity(0) == before
    monkeypatch.setattr(bench, "gpu_local_cpus", lambda i: None)
    with bench.near_gpu(0) as n:
        assert n.cpus is None and os.sched_getaffinity(0) == before
