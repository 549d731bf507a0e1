"""GPU parity of the per-triple association order, through the C ABI, against the fp64 oracle.

With TLR_ORDER_TRIPLE every tile triple (i, k, j) takes the cheaper side after
S_ikj = V_ik^T W_kj: U_ik (S_ikj Z_kj^T) when r_ik <= r_kj, else (U_ik S_ikj) Z_kj^T
("TLR Matrix Multiplication", section "The O_A O_B terms"). The product is the
same matrix as with the per-rectangle orders; only rounding differs. Checked
like the other orders: whole C, every output tile and every boundary region,
at 1e-2 (bf16) and 2.5e-3 (fp16), on the stated workloads, on unlike rank maps
where the sides really mix, with transposes and boundary tiles, with budgets
that split C, and at full size on sampled entries.
"""
import numpy as np
import pytest

import tlr_inputs as ti
from parity_check import check, interior_extents, tile_size
from test_parity_gpu import handle, run, sample_indices, torch_cuda  # noqa: F401

pytestmark = pytest.mark.gpu
TOL = {"bf16": 1e-2, "f16": 2.5e-3}
TRIPLE = 3


def check_p(out, ref, p, rows=None, cols=None):
    return check(out, ref, TOL[p.dtype], tile_size(p), rows, cols, regions=interior_extents(p), what=p.name)


def run_triple(p, handle, budget=None):
    out, info = run(p, handle, budget=budget, order=TRIPLE)
    assert info["runs_triple"] == info["runs"] >= 1
    return out, info


@pytest.mark.parametrize("cfg,scale,dtype", [(5, 8, None), (5, 4, None), (5, 8, "f16"), (5, 4, "f16")])
@pytest.mark.parametrize("variant", ["whole", "lowrank_only", "dense_only"])
def test_large_workload_family(oracle_lib, handle, cfg, scale, dtype, variant):
    kw = {}
    if variant == "lowrank_only":
        kw = dict(zero_diag=True, beta_override=0.0)
    elif variant == "dense_only":
        kw = dict(zero_lowrank=True)
    p = ti.problem(cfg, scale_down=scale, dtype_override=dtype, **kw)
    out, info = run_triple(p, handle)
    print(p.name, variant, check_p(out, oracle_lib.gemm_problem(p), p), info["runs"])


@pytest.mark.parametrize("n,budget", [(2048, None), (4096, None), (4096, 12 << 20), (4096, 3 << 20)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_unlike_rank_maps(oracle_lib, handle, n, budget, dtype):
    """Both sides in use within one output tile, one rectangle or many."""
    p = ti.asym_grid(n, 256, dtype)
    out, info = run_triple(p, handle, budget)
    if budget == 3 << 20:
        assert info["runs"] >= 8
    print(p.name, check_p(out, oracle_lib.gemm_problem(p), p), info["runs"])


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_pages_skewed_workload(oracle_lib, handle, dtype):
    p = ti.skewed_grid(4096, dtype)
    out, _ = run_triple(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("opA,opB", [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")])
def test_transposes_with_boundary(oracle_lib, handle, dtype, opA, opB):
    """A 72-wide boundary tile row and column (two panel parts per tile row), beta != 0."""
    rng = np.random.default_rng(41)
    N, b = 456, 128
    A = ti.make_tlr(rng, N, b, ti.rank_uniform(0, 40), dtype)
    B = ti.make_tlr(rng, N, b, ti.rank_uniform(0, 40), dtype)
    C = rng.standard_normal(N * N).astype(np.float32)
    p = ti.Problem("triple_transpose", A, B, opA, opB, 0.75, -1.25, C, N, N, dtype)
    out, _ = run_triple(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


def test_rank_extremes(oracle_lib, handle):
    """Rank-0 tiles (triples with no contribution), full-rank tiles, a tile row with no low-rank work."""
    rng = np.random.default_rng(42)
    N, b = 512, 64
    nt = N // b
    R = rng.integers(0, b + 1, size=(nt, nt))
    R[0, :] = 0
    R[:, 2] = b
    A = ti.make_tlr(rng, N, b, None, "bf16", ranks=R)
    B = ti.make_tlr(rng, N, b, None, "bf16", ranks=R.T.copy())
    p = ti.Problem("triple_ranks", A, B, "N", "N", 1.0, 0.0, None, N, N, "bf16")
    out, _ = run_triple(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


def test_alternating_sides_within_the_segment_limit(oracle_lib, handle):
    """The cheaper side alternates along k, so the planner regroups runs to fit a
    tile's K-loop; the product is unchanged."""
    n, b = 2048, 128
    nt = n // b
    ra = np.fromfunction(lambda i, k: np.where((k % 2) == 0, 8, 40), (nt, nt)).astype(np.int64)
    rb = np.fromfunction(lambda k, j: np.where((k % 2) == 0, 40, 8), (nt, nt)).astype(np.int64)
    rng = np.random.default_rng(43)
    A = ti.make_tlr(rng, n, b, None, "bf16", ranks=ra)
    B = ti.make_tlr(rng, n, b, None, "bf16", ranks=rb)
    p = ti.Problem("alternating", A, B, "N", "N", 1.0, 0.0, None, n, n, "bf16")
    out, _ = run_triple(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


def test_all_lowrank_rectangular_grid(oracle_lib, handle):
    """No dense tiles at all (the worked example's 2x3 by 3x3 grid of 256-tiles)."""
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")))
    rng = np.random.default_rng(44)
    A = ti.make_tlr(rng, 512, 256, None, "bf16", cols=768, diag_dense=False, ranks=np.array(g["rA"]))
    B = ti.make_tlr(rng, 768, 256, None, "bf16", diag_dense=False, ranks=np.array(g["rB_solutions"][1]))
    p = ti.Problem("triple_worked", A, B, "N", "N", 1.0, 0.0, None, 512, 768, "bf16")
    out, _ = run_triple(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


@pytest.mark.parametrize("variant", ["whole", "lowrank_only"])
def test_large_workload_full_size_sampled(oracle_lib, handle, variant):
    """N = 32768 with the 2 GiB budget, in the launch configuration the benchmark times."""
    kw = dict(zero_diag=True, beta_override=0.0) if variant == "lowrank_only" else {}
    p = ti.problem(5, **kw)
    out, info = run_triple(p, handle)
    rows = sample_indices(p.m, p.A.b, seed=5)
    cols = sample_indices(p.n, p.A.b, seed=15)
    ref = oracle_lib.gemm_problem(p, rows, cols)
    print(p.name, variant, check_p(out[np.ix_(rows, cols)], ref, p, rows, cols), info["runs"])
