"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle.

Tolerances (relative Frobenius norm): 2e-3 for fp32 inputs on TF32 tensor
cores, 1e-2 for bf16 inputs with fp32 accumulation. Each comparison holds for the
whole compared block, for every output tile of C on its own and, for products
with a boundary tile, for each of the four output regions (`parity_check`). The
dense diagonal terms dominate ||C|| in these workloads, so every workload is also
run term-isolated on the same seeded factors (dense tiles zeroed with beta = 0,
or low-rank factors zeroed), each against its own norm.
"""
import numpy as np
import pytest

import tlr_inputs as ti
from parity_check import check, interior_extents, rel, tile_size

pytestmark = pytest.mark.gpu
TOL = {"f32": 2e-3, "bf16": 1e-2}


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


@pytest.fixture(scope="module")
def handle(torch_cuda):
    import gemm_tlr_gb300 as g
    h = g.tlr_create(torch_cuda.cuda.current_stream().cuda_stream)
    yield h
    g.tlr_destroy(h)


def check_p(out, ref, p, tol=None, rows=None, cols=None):
    """Whole, per-tile and per-region parity of a product's C (or of sampled rows x cols of it)."""
    return check(out, ref, TOL[p.dtype] if tol is None else tol, tile_size(p), rows, cols,
                 regions=interior_extents(p), what=p.name)


def run(p, handle, budget=None, order=0, times=1):
    import gemm_tlr_gb300 as g
    from gemm_tlr_gb300.device import DeviceProblem
    dp = DeviceProblem(p)
    try:
        dp.make_plan(handle, budget, order)
        outs = []
        for _ in range(times):
            dp.reset_c()
            dp.run()
            assert g.tlr_get_device_status(handle) == 0
            outs.append(dp.result())
        return (outs if times > 1 else outs[0]), dp.info()
    finally:
        dp.close()


def sample_indices(n, b, per_tile=8, seed=0):
    """Rows of every tile (first, last and per_tile - 2 random ones) plus the
    matrix edges: with 8 a side every output tile's error is measured on about
    64 entries, enough for the per-tile check to be stable."""
    rng = np.random.default_rng(seed)
    idx = set()
    for t0 in range(0, n, b):
        t1 = min(n, t0 + b)
        idx.update({t0, t1 - 1})
        idx.update(int(x) for x in rng.integers(t0, t1, size=max(0, per_tile - 2)))
    idx.update({0, n - 1})
    return np.array(sorted(idx))


FULL_ORACLE_CASES = [(1, 1), (2, 4), (2, 1), (3, 8), (3, 4), (4, 16), (4, 8), (5, 16), (5, 8)]


@pytest.mark.parametrize("cfg,scale", FULL_ORACLE_CASES)
@pytest.mark.parametrize("variant", ["whole", "lowrank_only", "dense_only"])
def test_whole_product_matches_oracle(oracle_lib, handle, cfg, scale, variant):
    kw = {}
    if variant == "lowrank_only":
        kw = dict(zero_diag=True, beta_override=0.0)
    elif variant == "dense_only":
        kw = dict(zero_lowrank=True)
    p = ti.problem(cfg, scale_down=scale, **kw)
    out, info = run(p, handle)
    ref = oracle_lib.gemm_problem(p)
    res = check_p(out, ref, p)
    print(f"{p.name} {variant}: {res} (runs={info['runs']}, left={info['runs_left']})")


@pytest.mark.parametrize("cfg,order", [(2, 0), (3, 0), (4, 0), (5, 0), (5, 4)], ids=["2", "3", "4", "5", "5-per_rect"])
@pytest.mark.parametrize("variant", ["whole", "lowrank_only"])
def test_full_size_sampled(oracle_lib, handle, cfg, order, variant):
    """The graded sizes, in the launch configuration the benchmark times (and, for
    the large product, with the per-rectangle orders too), on sampled entries."""
    kw = dict(zero_diag=True, beta_override=0.0) if variant == "lowrank_only" else {}
    p = ti.problem(cfg, **kw)
    out, info = run(p, handle, order=order)
    b = p.A.b
    rows = sample_indices(p.m, b, seed=cfg)
    cols = sample_indices(p.n, b if p.B.kind == "tlr" else 1024, seed=cfg + 10)
    ref = oracle_lib.gemm_problem(p, rows, cols)
    got = out[np.ix_(rows, cols)]
    res = check_p(got, ref, p, rows=rows, cols=cols)
    print(f"{p.name} {variant} sampled: {res}")
    if cfg == 5 and order == 4:
        assert info["runs"] >= 2 and info["runs_triple"] == 0   # the 2 GiB budget forces a split
    elif cfg == 5:
        assert info["runs_triple"] == info["runs"]              # the default takes the per-triple order


@pytest.mark.parametrize("scale", [16, 8])
@pytest.mark.parametrize("variant", ["whole", "lowrank_only", "dense_only"])
def test_per_rectangle_orders_on_the_large_family(oracle_lib, handle, scale, variant):
    """The per-rectangle orders (TLR_ORDER_PER_RECT), which the default no longer
    takes for this family, against the oracle."""
    kw = {}
    if variant == "lowrank_only":
        kw = dict(zero_diag=True, beta_override=0.0)
    elif variant == "dense_only":
        kw = dict(zero_lowrank=True)
    p = ti.problem(5, scale_down=scale, **kw)
    out, info = run(p, handle, order=4)
    assert info["runs_triple"] == 0
    print(p.name, variant, check_p(out, oracle_lib.gemm_problem(p), p), info["runs"], info["runs_left"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("opA,opB", [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")])
def test_transposes_with_boundary(oracle_lib, handle, dtype, opA, opB):
    rng = np.random.default_rng(21)
    N, b = 456, 128            # 3 full tiles + a 72-wide boundary tile
    A = ti.make_tlr(rng, N, b, ti.rank_uniform(0, 40), dtype)
    B = ti.make_tlr(rng, N, b, ti.rank_uniform(0, 40), dtype)
    C = rng.standard_normal(N * N).astype(np.float32)
    p = ti.Problem("transpose", A, B, opA, opB, 0.75, -1.25, C, N, N, dtype)
    out, _ = run(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


@pytest.mark.parametrize("order", [1, 2])
def test_both_association_orders(oracle_lib, handle, order):
    p = ti.problem(2, scale_down=4)
    out, info = run(p, handle, order=order)
    assert (info["runs_left"] > 0) == (order == 2)
    check_p(out, oracle_lib.gemm_problem(p), p)


def test_small_budget_many_rectangles(oracle_lib, handle):
    import gemm_tlr_gb300 as g
    from gemm_tlr_gb300.device import host_descriptor
    p = ti.problem(5, scale_down=8)
    A, ka = host_descriptor(p.A)
    B, kb = host_descriptor(p.B)
    budget = g.tlr_gemm_workspace_bytes(0, 0, 0, A, B, 6)
    out, info = run(p, handle, budget=budget)
    assert 2 <= info["runs"] <= 6
    check_p(out, oracle_lib.gemm_problem(p), p)


@pytest.mark.parametrize("runs", [1, 6])
def test_merged_two_arena_schedule(oracle_lib, handle, monkeypatch, runs):
    """The single merged launch of CTA pairs, where Stages 1-2 of rectangle r + 1 run
    interleaved with the final products of rectangle r in a second arena."""
    import gemm_tlr_gb300 as g
    from gemm_tlr_gb300.device import host_descriptor
    monkeypatch.setenv("TLR_HYBRID", "0")
    p = ti.problem(5, scale_down=8)
    A, ka = host_descriptor(p.A)
    B, kb = host_descriptor(p.B)
    budget = g.tlr_gemm_workspace_bytes(0, 0, 0, A, B, runs)
    out, info = run(p, handle, budget=budget)
    assert (info["runs"] == 1) == (runs == 1)
    check_p(out, oracle_lib.gemm_problem(p), p)


@pytest.mark.parametrize("cfg,scale", [(5, 4), (3, 2), (2, 1)])
def test_single_cta_tiles_match_oracle(oracle_lib, handle, monkeypatch, cfg, scale):
    """128-row tiles on single CTAs (cta_group::1) for products whose default is CTA pairs."""
    monkeypatch.setenv("TLR_PAIR", "1")
    p = ti.problem(cfg, scale_down=scale)
    out, info = run(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


def test_rank_extremes(oracle_lib, handle):
    """Rank-0 tiles, full-rank tiles and a tile row with no low-rank work at all."""
    rng = np.random.default_rng(22)
    N, b = 384, 64
    nt = N // b
    R = rng.integers(0, b + 1, size=(nt, nt))
    R[0, :] = 0
    R[:, 2] = b
    A = ti.make_tlr(rng, N, b, None, "f32", ranks=R)
    B = ti.make_tlr(rng, N, b, None, "f32", ranks=R.T.copy())
    p = ti.Problem("ranks", A, B, "N", "N", 1.0, 0.0, None, N, N, "f32")
    out, _ = run(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


def test_ragged_tiles_smaller_than_mma_tile(oracle_lib, handle):
    rng = np.random.default_rng(23)
    N, b = 296, 96             # 96-row tiles (< 128) and an 8-row boundary
    A = ti.make_tlr(rng, N, b, ti.rank_uniform(1, 30), "bf16")
    B = ti.make_tlr(rng, N, b, ti.rank_uniform(1, 30), "bf16")
    p = ti.Problem("ragged", A, B, "N", "N", 1.0, 0.0, None, N, N, "bf16")
    out, _ = run(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


def test_all_lowrank_rectangular_grid(oracle_lib, handle):
    """The worked example's structure: a 2x3 by 3x3 grid of 256-tiles, no dense tiles."""
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")))
    rng = np.random.default_rng(24)
    A = ti.make_tlr(rng, 512, 256, None, "bf16", cols=768, diag_dense=False, ranks=np.array(g["rA"]))
    B = ti.make_tlr(rng, 768, 256, None, "bf16", diag_dense=False, ranks=np.array(g["rB_solutions"][0]))
    p = ti.Problem("worked", A, B, "N", "N", 1.0, 0.0, None, 512, 768, "bf16")
    out, info = run(p, handle, order=4)      # per rectangle: the right order, as the pages' example
    assert info["runs_right"] == 1 and info["runs_left"] == 0
    check_p(out, oracle_lib.gemm_problem(p), p)


def test_dense_left_operand(oracle_lib, handle):
    rng = np.random.default_rng(25)
    A = ti.make_dense(rng, 320, 512, "bf16")
    B = ti.make_tlr(rng, 512, 128, ti.rank_uniform(4, 48), "bf16")
    p = ti.Problem("dense_x_tlr", A, B, "N", "N", 1.0, 0.0, None, 320, 512, "bf16")
    out, info = run(p, handle)
    assert info["runs_left"] == info["runs"]
    check_p(out, oracle_lib.gemm_problem(p), p)


def test_alpha_zero_and_beta_zero(oracle_lib, handle, torch_cuda):
    p = ti.problem(1, beta_override=0.5, alpha_override=0.0)
    out, _ = run(p, handle)
    assert np.array_equal(out, 0.5 * p.C.astype(np.float64).reshape(p.n, p.m).T.astype(np.float32).astype(np.float64))
    p = ti.problem(1)                     # beta = 0 with C full of NaN
    out, _ = run(p, handle)
    assert np.isfinite(out).all()


def test_repeat_is_bitwise_deterministic(handle):
    p = ti.problem(2, scale_down=4)
    outs, _ = run(p, handle, times=2)
    assert np.array_equal(outs[0], outs[1])


def test_one_shot_entry_point(oracle_lib, handle, torch_cuda):
    import gemm_tlr_gb300 as g
    from gemm_tlr_gb300.device import DeviceProblem
    p = ti.problem(1)
    dp = DeviceProblem(p)
    need = g.tlr_gemm_workspace_bytes(handle, dp.opA, dp.opB, dp.A.desc, dp.B.desc, 1)
    ws = torch_cuda.empty(need, dtype=torch_cuda.uint8, device="cuda")
    g.tlr_gemm(handle, dp.opA, dp.opB, p.alpha, dp.A.desc, dp.B.desc, p.beta, dp.C.data_ptr(), p.m,
               ws.data_ptr(), need)
    assert g.tlr_get_device_status(handle) == 0
    check_p(dp.result(), oracle_lib.gemm_problem(p), p)


def test_host_buffers_are_refused_before_any_launch(handle, torch_cuda):
    """Operands, workspace and C must be device memory; a pinned host buffer is
    refused by plan creation or execution on the host (nothing is launched)."""
    import gemm_tlr_gb300 as g
    from gemm_tlr_gb300._abi import TLRError
    from gemm_tlr_gb300.device import DeviceProblem
    p = ti.problem(1)
    dp = DeviceProblem(p)
    try:
        host_u = dp.A.host["U"].pin_memory()
        saved = dp.A.desc.U
        dp.A.desc.U = host_u.data_ptr()
        with pytest.raises(TLRError) as e:
            dp.make_plan(handle)
        assert e.value.code == 1
        dp.A.desc.U = saved
        dp.make_plan(handle)
        host_c = torch_cuda.empty(p.m * p.n, dtype=torch_cuda.float32).pin_memory()
        with pytest.raises(TLRError) as e:
            g.tlr_plan_execute(dp.plan, p.alpha, p.beta, host_c.data_ptr(), p.m)
        assert e.value.code == 1
        dp.run()
        assert g.tlr_get_device_status(handle) == 0
    finally:
        dp.close()


def test_bounded_wait_reports_timeout_and_recovers(oracle_lib, handle):
    import gemm_tlr_gb300 as g
    g.tlr_set_wait_limit_us(handle, 200_000)
    g.tlr_debug_unsatisfied_wait(handle)
    assert g.tlr_get_device_status(handle) == 6          # TLR_STATUS_TIMEOUT
    g.tlr_set_wait_limit_us(handle, 2_000_000)
    assert g.tlr_get_device_status(handle) == 0          # cleared
    p = ti.problem(1)
    out, _ = run(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


def test_kernel_timing_counts_launches(handle):
    import gemm_tlr_gb300 as g
    g.tlr_reset_timing(handle)
    g.tlr_set_timing(handle, True)
    p = ti.problem(1)
    run(p, handle)
    ms, n = g.tlr_get_timing(handle, 5)
    g.tlr_set_timing(handle, False)
    assert n >= 1 and ms > 0


def test_two_launch_schedule_times_both_classes(oracle_lib, handle):
    """Final tiles on CTA pairs: each rectangle runs a Stages 1-2 launch (class 1)
    and a final-product launch (class 2); the result still matches the oracle."""
    import gemm_tlr_gb300 as g
    g.tlr_reset_timing(handle)
    g.tlr_set_timing(handle, True)
    p = ti.problem(5, scale_down=4)
    out, info = run(p, handle)
    (ms1, n1), (ms2, n2), (_, n5) = (g.tlr_get_timing(handle, k) for k in (1, 2, 5))
    g.tlr_set_timing(handle, False)
    assert n5 == 0 and n1 == info["runs"] and n2 == info["runs"] and ms1 > 0 and ms2 > 0
    check_p(out, oracle_lib.gemm_problem(p), p)
