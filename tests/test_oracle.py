"""Pins for the CPU fp64 oracle (no GPU).

Each test checks the oracle against something other than itself: brute force on
tiny inputs (dense reconstruction from the generator's own tile list, product by
numpy), closed forms, special cases, the transpose identity of the storage, and
the printed values of the worked example. ``test_planted_mistakes_are_caught``
builds copies of the oracle with known mistakes and shows the pins fail on each.
"""
import json
import os

import numpy as np
import pytest

import tlr_inputs as ti

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dense_from_tiles(X, op="N"):
    """Brute-force dense matrix from the generator's per-tile list (numpy)."""
    rd, cd = X.rdims, X.cdims
    M = np.zeros((X.rows, X.cols))
    r0, c0 = np.cumsum([0] + rd), np.cumsum([0] + cd)
    for (i, k), t in X.tiles.items():
        blk = t[1].astype(np.float64) if t[0] == "dense" else t[1].astype(np.float64) @ t[2].astype(np.float64).T
        M[r0[i]:r0[i + 1], c0[k]:c0[k + 1]] = blk
    return M.T if op == "T" else M


def brute(A, B, opA, opB, alpha, beta, C):
    Ad = dense_from_tiles(A, opA) if A.kind == "tlr" else None
    if B.kind == "tlr":
        Bd = dense_from_tiles(B, opB)
    else:
        Bd = B.data.astype(np.float64).reshape(B.rows, B.cols, order="F")
        Bd = Bd.T if opB == "T" else Bd
    out = alpha * Ad @ Bd
    if beta != 0.0:
        out += beta * C.astype(np.float64).reshape(out.shape[1], out.shape[0]).T
    return out


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


CASES = [(64, 16), (100, 32), (200, 64)]   # 100 and 200 have a ragged boundary tile


@pytest.mark.parametrize("N,b", CASES)
@pytest.mark.parametrize("opA,opB", [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")])
def test_oracle_matches_brute_force(oracle_lib, N, b, opA, opB):
    rng = np.random.default_rng(N * 7 + b)
    A = ti.make_tlr(rng, N, b, ti.rank_uniform(0, 9), "f32", keep_tiles=True)
    B = ti.make_tlr(rng, N, b, ti.rank_uniform(0, 9), "f32", keep_tiles=True)
    C = rng.standard_normal(N * N).astype(np.float32)
    out = oracle_lib.gemm_block(A, B, opA, opB, 1.25, -0.5, C, N, np.arange(N), np.arange(N))
    assert rel(out, brute(A, B, opA, opB, 1.25, -0.5, C)) < 1e-13


def test_oracle_rectangular_all_lowrank_grid(oracle_lib):
    """No dense diagonal, rectangular grids (the worked example's structure)."""
    rng = np.random.default_rng(5)
    A = ti.make_tlr(rng, 64, 32, ti.rank_uniform(1, 8), "f32", cols=96, diag_dense=False, keep_tiles=True)
    B = ti.make_tlr(rng, 96, 32, ti.rank_uniform(1, 8), "f32", diag_dense=False, keep_tiles=True)
    out = oracle_lib.gemm_block(A, B, "N", "N", 1.0, 0.0, None, 64, np.arange(64), np.arange(96))
    assert rel(out, brute(A, B, "N", "N", 1.0, 0.0, None)) < 1e-13


def test_oracle_dense_right_operand(oracle_lib):
    rng = np.random.default_rng(6)
    A = ti.make_tlr(rng, 128, 32, ti.rank_uniform(1, 16), "bf16", keep_tiles=True)
    B = ti.make_dense(rng, 128, 40, "bf16")
    out = oracle_lib.gemm_block(A, B, "N", "N", 0.75, 0.0, None, 128, np.arange(128), np.arange(40))
    assert rel(out, brute(A, B, "N", "N", 0.75, 0.0, None)) < 1e-13


def _full_rank_tlr(rng, Md, b):
    """TLR storage of a dense matrix with U_ij = M_ij and V_ij = I (rank b)."""
    N = Md.shape[0]
    X = ti.make_tlr(rng, N, b, ti.rank_fixed(b), "f32", keep_tiles=True)
    for (i, k), t in X.tiles.items():
        blk = Md[i * b:(i + 1) * b, k * b:(k + 1) * b]
        if t[0] == "dense":
            t[1][...] = blk
        else:
            t[1][...] = blk
            t[2][...] = np.eye(b, dtype=np.float32)
    return X


def test_full_rank_tlr_equals_dense_product(oracle_lib):
    rng = np.random.default_rng(7)
    N, b = 96, 32
    Ad = rng.standard_normal((N, N)).astype(np.float32)
    Bd = rng.standard_normal((N, N)).astype(np.float32)
    A, B = _full_rank_tlr(rng, Ad, b), _full_rank_tlr(rng, Bd, b)
    out = oracle_lib.gemm_block(A, B, "N", "N", 1.0, 0.0, None, N, np.arange(N), np.arange(N))
    ref = Ad.astype(np.float64) @ Bd.astype(np.float64)
    assert rel(out, ref) < 1e-14


def test_closed_form_constant_rank_one_tiles(oracle_lib):
    """A_ik = a_ik * 1 1^T (rank one), dense tiles a_ii * 1 1^T; C = b * (a @ c) (x) 1 1^T."""
    rng = np.random.default_rng(8)
    N, b = 96, 32
    nt = N // b
    a = rng.integers(-4, 5, size=(nt, nt)).astype(np.float64)
    c = rng.integers(-4, 5, size=(nt, nt)).astype(np.float64)
    mats = []
    for coef in (a, c):
        X = ti.make_tlr(rng, N, b, ti.rank_fixed(1), "f32", keep_tiles=True)
        for (i, k), t in X.tiles.items():
            if t[0] == "dense":
                t[1][...] = coef[i, k]
            else:
                t[1][...] = coef[i, k]
                t[2][...] = 1.0
        mats.append(X)
    out = oracle_lib.gemm_block(mats[0], mats[1], "N", "N", 2.0, 0.0, None, N, np.arange(N), np.arange(N))
    ref = 2.0 * b * np.kron(a @ c, np.ones((b, b)))
    assert np.array_equal(out, ref)


def test_alpha_zero_gives_beta_c_and_reads_no_operand(oracle_lib):
    rng = np.random.default_rng(9)
    N, b = 64, 16
    A = ti.make_tlr(rng, N, b, ti.rank_fixed(4), "f32")
    B = ti.make_tlr(rng, N, b, ti.rank_fixed(4), "f32")
    A.U[:] = np.nan
    B.D[:] = np.nan
    C = rng.standard_normal(N * N).astype(np.float32)
    out = oracle_lib.gemm_block(A, B, "N", "N", 0.0, 0.5, C, N, np.arange(N), np.arange(N))
    assert np.array_equal(out, 0.5 * C.astype(np.float64).reshape(N, N).T)


def test_beta_zero_does_not_read_c(oracle_lib):
    rng = np.random.default_rng(10)
    N, b = 64, 16
    A = ti.make_tlr(rng, N, b, ti.rank_fixed(4), "f32")
    B = ti.make_tlr(rng, N, b, ti.rank_fixed(4), "f32")
    Cnan = np.full(N * N, np.nan, dtype=np.float32)
    out = oracle_lib.gemm_block(A, B, "N", "N", 1.0, 0.0, Cnan, N, np.arange(N), np.arange(N))
    ref = oracle_lib.gemm_block(A, B, "N", "N", 1.0, 0.0, None, N, np.arange(N), np.arange(N))
    assert np.isfinite(out).all() and np.array_equal(out, ref)


def _explicit_transpose(X):
    """TLR storage of X^T built by swapping the factor families (role swap)."""
    Y = ti.TLRMatrix(rows=X.cols, cols=X.rows, b=X.b, diag_dense=X.diag_dense,
                     ranks=np.ascontiguousarray(X.ranks.T), dtype=X.dtype,
                     U=X.V.copy(), V=X.U.copy())
    b = X.b
    if X.D is not None:
        Y.D = X.D.reshape(-1, b, b).transpose(0, 2, 1).copy().reshape(-1)  # each tile transposed
    if X.gamma is not None:
        r = X.rows % b
        Y.bu_U, Y.bu_V, Y.bv_U, Y.bv_V = X.bv_V.copy(), X.bv_U.copy(), X.bu_V.copy(), X.bu_U.copy()
        Y.gamma = X.gamma.reshape(r, r).T.copy().reshape(-1)
    return Y


@pytest.mark.parametrize("N,b", [(96, 32), (200, 64)])
def test_transpose_identity(oracle_lib, N, b):
    """(A^T)_ik = V_ki U_ki^T: op(A)=T equals the role-swapped storage with op N."""
    rng = np.random.default_rng(11)
    A = ti.make_tlr(rng, N, b, ti.rank_uniform(1, 9), "f32", keep_tiles=True)
    B = ti.make_tlr(rng, N, b, ti.rank_uniform(1, 9), "f32")
    At = _explicit_transpose(A)
    o1 = oracle_lib.gemm_block(A, B, "T", "N", 1.0, 0.0, None, N, np.arange(N), np.arange(N))
    o2 = oracle_lib.gemm_block(At, B, "N", "N", 1.0, 0.0, None, N, np.arange(N), np.arange(N))
    assert np.array_equal(o1, o2)
    assert rel(oracle_lib.expand_tile(A, 1, 0, "T"), dense_from_tiles(A, "T")[b:2 * b, 0:b]) < 1e-15


def test_sampled_block_equals_full(oracle_lib):
    p = ti.problem(2, scale_down=8)
    full = oracle_lib.gemm_problem(p)
    rows = np.array([0, 5, 31, 100, p.m - 1])
    cols = np.array([1, 64, 77, p.n - 1])
    assert np.array_equal(oracle_lib.gemm_problem(p, rows, cols), full[np.ix_(rows, cols)])


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_evaluation_orders_agree(oracle_lib, cfg):
    """Per-k loop and fused-k three-stage order give the definition's result (fp64)."""
    from oracle import orders
    p = ti.problem(cfg, scale_down={1: 1, 2: 8, 3: 8, 4: 16, 5: 32}[cfg])
    d = oracle_lib.gemm_problem(p)
    k = orders.kblas_order(p.A, p.B, p.opA, p.opB, p.alpha, p.beta, p.C, p.m)
    f = orders.fused_k_order(p.A, p.B, p.opA, p.opB, p.alpha, p.beta, p.C, p.m)
    assert rel(k, d) < 1e-12
    assert rel(f, d) < 1e-12


def test_worked_example_metadata():
    from oracle import planner_ref
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    b, pr = g["b"], g["printed"]
    for rB in g["rB_solutions"]:
        md = planner_ref.metadata(g["rA"], rB, [b, b], [b, b, b], [b, b, b])
        assert md["rho"] == pr["rho"] and md["gamma"] == pr["gamma"]
        assert md["F_R"] == 2 * b * b * pr["F_R_over_2b2"]
        assert md["F_L"] == 2 * b * b * pr["F_L_over_2b2"]
        assert round(100 * (1 - md["F_R"] / md["F_L"])) == pr["right_saving_percent_about"]
        assert [list(s) for s in md["stage1"]] == pr["stage1_shapes"]
        assert md["coupling_products"] == pr["coupling_products"]
        assert md["distinct_shapes"] == pr["distinct_shapes"]
        assert list(md["T_R"]) == pr["T_R"] and list(md["T_L"]) == pr["T_L"]
        assert [list(s) for s in md["stage3_R"]] == pr["stage3_shapes"]
        assert md["order"] == pr["order"]
        assert [md["rho"][0], 3 * b] == pr["T1_shape"]


def test_oracle_rejects_bad_ranks(oracle_lib):
    rng = np.random.default_rng(12)
    A = ti.make_tlr(rng, 64, 16, ti.rank_fixed(4), "f32")
    A.ranks[0, 1] = 17                      # larger than the tile
    assert oracle_lib.check(A) != 0


@pytest.mark.parametrize("code", [1, 2, 3, 4])
def test_planted_mistakes_are_caught(oracle_lib, tmp_path, code):
    """Copies of the oracle with a planted mistake fail the brute-force pin."""
    path = oracle_lib.load_mutant(code, str(tmp_path))
    rng = np.random.default_rng(13)
    N, b = 100, 32
    A = ti.make_tlr(rng, N, b, ti.rank_uniform(2, 9), "f32", keep_tiles=True)
    B = ti.make_tlr(rng, N, b, ti.rank_uniform(2, 9), "f32", keep_tiles=True)
    C = rng.standard_normal(N * N).astype(np.float32)
    ref = brute(A, B, "N", "N", 1.0, 0.5, C)
    with oracle_lib.use_library(path):
        out = oracle_lib.gemm_block(A, B, "N", "N", 1.0, 0.5, C, N, np.arange(N), np.arange(N))
    assert rel(out, ref) > 1e-3


def test_f16_rounding_is_nearest_even():
    """fp16 inputs: 10 stored mantissa bits, ties to even (checked on exact ties)."""
    one = np.float32(1.0)
    x = np.array([1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, -(1 + 2.0 ** -11), 65504.0, 2.0 ** -24], dtype=np.float32)
    got = ti.f16_round(x)
    assert got[0] == one                      # tie between 1 and 1 + 2^-10: the even one
    assert got[1] == np.float32(1 + 2.0 ** -9)  # tie between 1 + 2^-10 and 1 + 2^-9: the even one
    assert got[2] == -one
    assert got[3] == np.float32(65504.0)      # largest finite fp16
    assert got[4] == np.float32(2.0 ** -24)   # smallest subnormal survives
    p = ti.skewed_grid(1024, "f16")
    for a in (p.A.U, p.A.V, p.A.D, p.B.U):
        assert np.array_equal(a, a.astype(np.float16).astype(np.float32))


def test_skewed_ranks_stay_in_range_and_lean_low():
    """The pages' second workload: 8 x 8 tiles, ranks on [b/32, b/16], skewed towards b/32."""
    p = ti.skewed_grid(8192, "f32")
    b = p.A.b
    assert b == 1024 and p.A.ranks.shape == (8, 8)
    for X in (p.A, p.B):
        off = X.ranks[~np.eye(8, dtype=bool)]
        assert off.min() >= b // 32 and off.max() <= b // 16
        assert np.all(np.diag(X.ranks) == 0)            # dense diagonal
    r = ti.rank_skewed(256, 512)(np.random.default_rng(0), 200, 200, None, None)
    assert r.min() == 256 and r.max() == 512
    assert abs(r.mean() - (256 + 257 / 3)) < 2.0          # E[lo + (hi-lo+1) u^2] = lo + (hi-lo+1)/3
    assert np.median(r) < 256 + 257 / 2                   # more mass below the midpoint
    q = ti.skewed_grid(8192, "f32")
    assert np.array_equal(q.A.ranks, p.A.ranks)           # seeded


def test_oracle_matches_brute_force_on_fp16_skewed_grid(oracle_lib):
    """fp16 inputs on the 8 x 8 skewed-rank grid: oracle against a numpy product of the
    dense reconstruction (every value is fp16-exact, so the check is dtype-independent)."""
    p = ti.skewed_grid(512, "f16", keep_tiles=True)
    ref = dense_from_tiles(p.A) @ dense_from_tiles(p.B)
    got = oracle_lib.gemm_problem(p)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))
