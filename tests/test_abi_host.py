"""C-ABI library on the host (no GPU): symbols, planner metadata, validation, plan tables.

The planner is pinned by the worked example's printed values ("Tile-Low-Rank
GEMM: Designing Storage Around the Contraction", sections "One product, three
stages" and "Association order and workspace") and cross-checked against the
oracle's own metadata definitions on random rank maps. The table validator
(`tlr_debug_check_plan`) proves, without a GPU, that every plan's TMA views and
output writes stay inside their buffers and that every dependency is satisfied.
"""
import ctypes
import functools
import json
import os

import numpy as np
import pytest

import tlr_inputs as ti

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def g():
    from gemm_tlr_gb300.build import build
    build()
    import gemm_tlr_gb300
    gemm_tlr_gb300.lib()
    return gemm_tlr_gb300


def desc(ranks, rows, cols, b, diag_dense=0, dtype=1):
    import gemm_tlr_gb300._abi as abi
    d = abi.tlr_operand_t()
    r = np.ascontiguousarray(ranks, dtype=np.int32)
    d.kind, d.dtype, d.rows, d.cols, d.b, d.diag_dense, d.ranks = 0, dtype, rows, cols, b, diag_dense, r.ctypes.data
    return d, r


def test_library_exports_every_declared_symbol(g):
    L = ctypes.CDLL(g._abi.LIB_PATH)
    names = g.header_symbols()
    assert len(names) >= 18
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(g):
    assert g.tlr_status_string(0) == "TLR_STATUS_OK"
    assert g.tlr_status_string(6) == "TLR_STATUS_TIMEOUT"


def test_create_without_gpu_reports_not_initialized(g):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(g.TLRError) as e:
        g.tlr_create(0)
    assert e.value.code == 7


@pytest.mark.parametrize("sol", [0, 1])
def test_planner_matches_worked_example(g, sol):
    gold = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    b, pr = gold["b"], gold["printed"]
    A, ka = desc(gold["rA"], 2 * b, 3 * b, b)
    B, kb = desc(gold["rB_solutions"][sol], 3 * b, 3 * b, b)
    out = g.tlr_analyze(0, 0, A, B, 2, 3, 3)
    assert list(out["rho"]) == pr["rho"] and list(out["gamma"]) == pr["gamma"]
    assert out["F_R"] == 2 * b * b * pr["F_R_over_2b2"] and out["F_L"] == 2 * b * b * pr["F_L_over_2b2"]
    assert out["stage1_mnk"].reshape(-1, 3).tolist() == pr["stage1_shapes"]
    assert out["stage3_mnk"].reshape(-1, 3).tolist() == pr["stage3_shapes"]
    assert out["coupling_products"] == pr["coupling_products"]
    assert out["distinct_shapes"] == pr["distinct_shapes"]
    assert [out["T_right_rows"], out["T_right_cols"]] == pr["T_R"]
    assert [out["T_left_rows"], out["T_left_cols"]] == pr["T_L"]
    assert out["order"] == (1 if pr["order"] == "R" else 2)


@pytest.mark.parametrize("seed", range(6))
def test_planner_matches_oracle_metadata_on_random_ranks(g, seed):
    from oracle import planner_ref
    rng = np.random.default_rng(seed)
    nI, nK, nJ, b = rng.integers(1, 6, size=3).tolist() + [64]
    rA = rng.integers(0, b + 1, size=(nI, nK))
    rB = rng.integers(0, b + 1, size=(nK, nJ))
    A, ka = desc(rA, nI * b, nK * b, b)
    B, kb = desc(rB, nK * b, nJ * b, b)
    out = g.tlr_analyze(0, 0, A, B, nI, nK, nJ)
    md = planner_ref.metadata(rA, rB, [b] * nI, [b] * nK, [b] * nJ)
    assert list(out["rho"]) == md["rho"] and list(out["gamma"]) == md["gamma"]
    assert list(out["sigma"]) == md["sigma"] and list(out["Gamma"]) == md["Gamma"]
    assert out["F_R"] == md["F_R"] and out["F_L"] == md["F_L"]
    assert out["coupling_products"] == md["coupling_products"]
    assert out["distinct_shapes"] == md["distinct_shapes"]


def test_invalid_descriptors_are_rejected_before_launch(g):
    from gemm_tlr_gb300.device import fake_descriptor
    rng = np.random.default_rng(1)
    X = ti.make_tlr(rng, 256, 64, ti.rank_fixed(8), "bf16")
    A, ka = fake_descriptor(X, 1 << 40)
    B, kb = fake_descriptor(X, 1 << 41)
    assert g.tlr_debug_check_plan(0, 0, A, B, 1 << 30)[0] == 0
    bad_rank = X.ranks.copy()
    bad_rank[0, 1] = 65                              # larger than the tile
    A2, k2 = desc(bad_rank, 256, 256, 64, 1)
    A2.U, A2.V, A2.D = A.U, A.V, A.D
    assert g.tlr_debug_check_plan(0, 0, A2, B, 1 << 30)[0] == 1
    A3, k3 = fake_descriptor(X, (1 << 40) + 8)      # base not 16-byte aligned
    assert g.tlr_debug_check_plan(0, 0, A3, B, 1 << 30)[0] == 2
    Y = ti.make_tlr(rng, 260, 65, ti.rank_fixed(8), "bf16")   # tile dimension not a multiple of 8
    A4, k4 = fake_descriptor(Y, 1 << 40)
    assert g.tlr_debug_check_plan(0, 0, A4, A4, 1 << 30)[0] == 2
    assert g.tlr_debug_check_plan(0, 0, A, B, 1024)[0] == 3          # workspace too small
    D = ti.make_dense(rng, 256, 256, "bf16")
    Dd, kd = fake_descriptor(D, 1 << 42)
    assert g.tlr_debug_check_plan(0, 0, Dd, Dd, 1 << 30)[0] == 4      # dense x dense unsupported
    F = ti.make_tlr(rng, 256, 64, ti.rank_fixed(8), "f32")
    Fd, kf = fake_descriptor(F, 1 << 42)
    assert g.tlr_debug_check_plan(0, 0, A, Fd, 1 << 30)[0] == 4       # mixed element types


def test_offsets_are_checked_against_prefix_sums(g):
    from gemm_tlr_gb300.device import fake_descriptor
    rng = np.random.default_rng(2)
    X = ti.make_tlr(rng, 256, 64, ti.rank_uniform(1, 8), "bf16")
    A, ka = fake_descriptor(X, 1 << 40)
    R = X.ranks.astype(np.int64)
    uoff = np.zeros_like(R)
    c = 0
    for i in range(4):
        for k in range(4):
            if i != k:
                uoff[i, k] = 64 * c
                c += R[i, k]
    uoff = np.ascontiguousarray(uoff.reshape(-1))
    A.u_offsets = uoff.ctypes.data
    assert g.tlr_debug_check_plan(0, 0, A, A, 1 << 30)[0] == 0
    uoff[6] += 64                              # tile (1, 2)
    assert g.tlr_debug_check_plan(0, 0, A, A, 1 << 30)[0] == 1


CASES = [(1, 1), (2, 1), (3, 1), (4, 1), (5, 1), (5, 8), (3, 8), (2, 4)]


@pytest.mark.parametrize("cfg,scale", CASES)
@pytest.mark.parametrize("order", [0, 1, 2])
def test_plan_tables_are_valid(g, cfg, scale, order):
    from gemm_tlr_gb300.device import fake_descriptor
    p = ti.problem(cfg, scale_down=scale)
    A, ka = fake_descriptor(p.A, 1 << 40)
    B, kb = fake_descriptor(p.B, 1 << 41)
    opA = 1 if p.opA == "T" else 0
    if cfg == 4 and order == 2:
        pytest.skip("a dense right operand has only the right order")
    budget = p.budget or g.tlr_gemm_workspace_bytes(0, opA, 0, A, B, 1)
    st, msg, info = g.tlr_debug_check_plan(opA, 0, A, B, budget, order)
    assert st == 0, msg
    from gemm_tlr_gb300 import flops
    rects = g.tlr_debug_plan_rects(opA, 0, A, B, budget, order)
    want = flops.executed_flops_rects(p, rects)["total"]
    assert abs(info["flops_executed"] - want) <= 1e-9 * want
    if cfg == 5 and scale == 1:
        assert info["workspace_bytes"] <= p.budget
        # the default takes the per-triple order in one rectangle; a single order needs a split
        assert info["runs"] >= 2 if order else info["runs_triple"] == info["runs"] == 1


def test_workspace_bytes_gives_the_requested_runs(g):
    from gemm_tlr_gb300.device import fake_descriptor
    p = ti.problem(5, scale_down=8)
    A, ka = fake_descriptor(p.A, 1 << 40)
    B, kb = fake_descriptor(p.B, 1 << 41)
    prev = None
    for runs in (1, 2, 3, 6):
        need = g.tlr_gemm_workspace_bytes(0, 0, 0, A, B, runs)
        st, msg, info = g.tlr_debug_check_plan(0, 0, A, B, need)
        assert st == 0 and info["runs"] <= max(runs, 1) and info["workspace_bytes"] <= need
        if prev is not None:
            assert need <= prev
        prev = need


def test_fp16_descriptors_plan_and_check_like_bf16(g):
    """fp16 operands: accepted, 16-byte rule on tile dimensions (d % 8), mixed 16-bit types rejected,
    and the plan tables of fp16 workloads pass the host-side proof."""
    from gemm_tlr_gb300.device import fake_descriptor
    rng = np.random.default_rng(3)
    X = ti.make_tlr(rng, 256, 64, ti.rank_fixed(8), "f16")
    A, ka = fake_descriptor(X, 1 << 40)
    B, kb = fake_descriptor(X, 1 << 41)
    assert A.dtype == g.TLR_F16
    assert g.tlr_debug_check_plan(0, 0, A, B, 1 << 30)[0] == 0
    Y = ti.make_tlr(rng, 260, 65, ti.rank_fixed(8), "f16")       # tile dimension not a multiple of 8
    Yd, ky = fake_descriptor(Y, 1 << 42)
    assert g.tlr_debug_check_plan(0, 0, Yd, Yd, 1 << 30)[0] == 2
    Z = ti.make_tlr(rng, 256, 64, ti.rank_fixed(8), "bf16")
    Zd, kz = fake_descriptor(Z, 1 << 42)
    assert g.tlr_debug_check_plan(0, 0, A, Zd, 1 << 30)[0] == 4       # fp16 x bf16: mixed element types
    for p in (ti.problem(5, scale_down=8, dtype_override="f16"), ti.problem(4, scale_down=8, dtype_override="f16"),
              ti.skewed_grid(2048, "f16")):
        Ad, ka2 = fake_descriptor(p.A, 1 << 40)
        Bd, kb2 = fake_descriptor(p.B, 1 << 44)
        ws = p.budget or g.tlr_gemm_workspace_bytes(0, 0, 0, Ad, Bd, 1)
        st, msg, info = g.tlr_debug_check_plan(0, 0, Ad, Bd, ws)
        assert st == 0, (p.name, msg)


@functools.lru_cache(maxsize=None)
def _problem(cfg, scale):
    return ti.problem(cfg, scale_down=scale)


SCHEDULES = [{}, {"TLR_HYBRID": "0"}, {"TLR_SPLIT_LAUNCHES": "1"}, {"TLR_L1_PAIR": "1"},
             {"TLR_L1_PAIR": "0"}, {"TLR_PAIR": "1"}, {"TLR_ARENAS": "1", "TLR_HYBRID": "0"},
             {"TLR_TRIPLE": "0"}, {"TLR_TRIPLE": "1"}, {"TLR_PIPELINE_ROWS": "0", "TLR_HYBRID": "0"},
             {"TLR_PIPELINE_ROWS": "2", "TLR_HYBRID": "0"}, {"TLR_PREP_BN": "128"},
             {"TLR_PREP_BN": "128", "TLR_L1_BN": "128"}, {"TLR_QUAD": "1"}]


@pytest.mark.parametrize("env", SCHEDULES, ids=lambda e: ",".join(f"{k}={v}" for k, v in e.items()) or "default")
@pytest.mark.parametrize("cfg,scale", [(5, 1), (5, 4), (4, 1), (3, 2)])
def test_every_schedule_variant_validates(g, monkeypatch, env, cfg, scale):
    """Each launch schedule the planner can build (defaults and tuning overrides)
    passes the host validator: views and writes in bounds, C covered once, T
    covered, and every dependency wait met by lower tickets of its own launch."""
    from gemm_tlr_gb300.device import fake_descriptor
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    p = _problem(cfg, scale)
    A, ka = fake_descriptor(p.A, 1 << 40)
    B, kb = fake_descriptor(p.B, 1 << 41)
    opA = 1 if p.opA == "T" else 0
    budget = p.budget or g.tlr_gemm_workspace_bytes(0, opA, 0, A, B, 1)
    st, msg, info = g.tlr_debug_check_plan(opA, 0, A, B, budget)
    assert st == 0, msg
    assert info["launches"] >= 1


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_plan_flops_recounted_rectangle_by_rectangle(g, cfg):
    """The planner's executed-FLOP figure equals an independent count from the
    ranks (gemm_tlr_gb300.flops) over the rectangles it reports, each with its
    own association order ("Tile-Low-Rank GEMM: Designing Storage Around the
    Contraction", section "Association order and workspace": the cheaper order
    per rectangle). The large product's 2 GiB plan mixes both orders."""
    from gemm_tlr_gb300 import flops as fl
    from gemm_tlr_gb300.device import fake_descriptor
    p = ti.problem(cfg)
    A, ka = fake_descriptor(p.A, 1 << 40)
    B, kb = fake_descriptor(p.B, 1 << 42)
    opA, opB = int(p.opA == "T"), int(p.opB == "T")
    budget = p.budget or (1 << 40)
    st, msg, info = g.tlr_debug_check_plan(opA, opB, A, B, budget)
    assert st == 0, msg
    rects = g.tlr_debug_plan_rects(opA, opB, A, B, budget)
    assert len(rects) == info["runs"]
    assert sum(r[4] == "L" for r in rects) == info["runs_left"]
    counted = fl.executed_flops_rects(p, rects)
    assert counted["total"] == pytest.approx(info["flops_executed"], rel=1e-12)
    for k, name in (("stage1", "flops_stage1"), ("stage2", "flops_stage2"), ("stage3", "flops_stage3"),
                    ("dense", "flops_dense_terms")):
        assert counted[k] == pytest.approx(info[name], rel=1e-12, abs=1.0)
    if cfg == 5:
        # the default takes the per-triple order here; the per-rectangle plan of the
        # 2 GiB budget mixes both orders, and either order over all of C gives the
        # right-order count of the survey table, 4.167e12
        assert {r[4] for r in rects} == {"P"}
        per = g.tlr_debug_plan_rects(opA, opB, A, B, budget, g.TLR_ORDER_PER_RECT)
        st, msg, pinfo = g.tlr_debug_check_plan(opA, opB, A, B, budget, g.TLR_ORDER_PER_RECT)
        assert st == 0, msg
        assert {r[4] for r in per} == {"R", "L"}
        mixed = fl.executed_flops_rects(p, per)["total"]
        assert mixed == pytest.approx(pinfo["flops_executed"], rel=1e-12)
        assert fl.executed_flops(p, "R")["total"] == pytest.approx(4.167e12, rel=1e-3)
        assert fl.executed_flops(p, "L")["total"] == pytest.approx(4.167e12, rel=1e-3)
        assert counted["total"] < mixed < fl.executed_flops(p, "R")["total"]
        forced = g.tlr_debug_plan_rects(opA, opB, A, B, budget, g.TLR_ORDER_RIGHT)
        assert {r[4] for r in forced} == {"R"}
        assert fl.executed_flops_rects(p, forced)["total"] == pytest.approx(fl.executed_flops(p, "R")["total"],
                                                                            rel=1e-12)


def _fake(p):
    from gemm_tlr_gb300.device import fake_descriptor
    A, ka = fake_descriptor(p.A, 1 << 40)
    B, kb = fake_descriptor(p.B, 1 << 42)
    return A, B, (ka, kb), int(p.opA == "T"), int(p.opB == "T")


TRIPLE_CASES = [("cfg5/8", lambda: ti.problem(5, scale_down=8), None),
                ("cfg5", lambda: ti.problem(5), None),
                ("asym", lambda: ti.asym_grid(2048, 256), None),
                ("asym_split", lambda: ti.asym_grid(4096, 256), 12 << 20),
                ("skewed", lambda: ti.skewed_grid(4096, "bf16"), None),
                ("f16_boundary_TN", lambda: ti.Problem(
                    "b", ti.make_tlr(np.random.default_rng(5), 456, 128, ti.rank_uniform(0, 40), "f16"),
                    ti.make_tlr(np.random.default_rng(6), 456, 128, ti.rank_uniform(0, 40), "f16"),
                    "T", "N", 1.0, 0.5, None, 456, 456, "f16"), None)]


@pytest.mark.parametrize("name,make,budget", TRIPLE_CASES, ids=[c[0] for c in TRIPLE_CASES])
def test_per_triple_plans_validate_and_count(g, name, make, budget):
    """The per-triple order ("TLR Matrix Multiplication", section "The O_A O_B
    terms": each (i, k, j) takes the side of min(r_ik, r_kj)) builds tables the
    host validator accepts (every view inside its buffer, C covered once, every
    terminal element a final product reads written exactly once), executes the
    FLOPs an independent count from the ranks gives, and never more than the
    per-rectangle plans."""
    from gemm_tlr_gb300 import flops as fl
    p = make()
    A, B, keep, opA, opB = _fake(p)
    budget = budget or p.budget or (1 << 40)
    st, msg, info = g.tlr_debug_check_plan(opA, opB, A, B, budget, g.TLR_ORDER_TRIPLE)
    assert st == 0, msg
    assert info["runs_triple"] == info["runs"] >= 1
    rects = g.tlr_debug_plan_rects(opA, opB, A, B, budget, g.TLR_ORDER_TRIPLE)
    assert {r[4] for r in rects} == {"P"}
    counted = fl.executed_flops_rects(p, rects)
    assert counted["total"] == pytest.approx(info["flops_executed"], rel=1e-12)
    assert counted["stage3"] == pytest.approx(info["flops_stage3"], rel=1e-12)
    st2, _, per = g.tlr_debug_check_plan(opA, opB, A, B, budget, g.TLR_ORDER_PER_RECT)
    assert st2 == 0 and info["flops_executed"] <= per["flops_executed"]
    if name == "cfg5":
        # the large product: final products 3.27e12 -> 1.59e12 FLOP
        assert info["flops_stage3"] == pytest.approx(1.595e12, rel=1e-3)
        assert per["flops_stage3"] == pytest.approx(3.265e12, rel=1e-3)


def test_four_orders_differ_on_the_asymmetric_workload(g):
    """Right, left, per-rectangle (a budget that splits C) and per-triple plans
    of the unlike-rank workload execute four different FLOP counts, each equal
    to the independent count over the plan's rectangles."""
    from gemm_tlr_gb300 import flops as fl
    p = ti.asym_grid(4096, 256)
    A, B, keep, opA, opB = _fake(p)
    seen = {}
    for budget in (1 << 40, 24 << 20, 12 << 20):
        for order in (g.TLR_ORDER_RIGHT, g.TLR_ORDER_LEFT, g.TLR_ORDER_PER_RECT, g.TLR_ORDER_TRIPLE):
            st, msg, info = g.tlr_debug_check_plan(opA, opB, A, B, budget, order)
            if st == 3:
                continue
            assert st == 0, msg
            rects = g.tlr_debug_plan_rects(opA, opB, A, B, budget, order)
            assert fl.executed_flops_rects(p, rects)["total"] == pytest.approx(info["flops_executed"], rel=1e-12)
            kinds = "".join(sorted({r[4] for r in rects}))
            seen.setdefault(kinds, set()).add(round(info["flops_executed"]))
    assert {"R", "L", "LR", "P"} <= set(seen), seen
    per = {k: min(v) for k, v in seen.items()}
    assert len(set(per.values())) == len(per)           # four different counts
    assert per["P"] < min(per["R"], per["L"], per["LR"])


def test_per_triple_order_needs_two_16_bit_tlr_operands(g):
    rng = np.random.default_rng(7)
    F = ti.make_tlr(rng, 256, 64, ti.rank_fixed(8), "f32")
    from gemm_tlr_gb300.device import fake_descriptor
    Fd, kf = fake_descriptor(F, 1 << 40)
    assert g.tlr_debug_check_plan(0, 0, Fd, Fd, 1 << 30, g.TLR_ORDER_TRIPLE)[0] == 4
    X = ti.make_tlr(rng, 256, 64, ti.rank_fixed(8), "bf16")
    D = ti.make_dense(rng, 256, 128, "bf16")
    Xd, kx = fake_descriptor(X, 1 << 40)
    Dd, kd = fake_descriptor(D, 1 << 42)
    assert g.tlr_debug_check_plan(0, 0, Xd, Dd, 1 << 30, g.TLR_ORDER_TRIPLE)[0] == 4


def test_per_triple_segment_limit_on_alternating_ranks(g):
    """Ranks that make the cheaper side alternate along k: every output tile's
    K-loop still fits the kernel's segment limit (the validator checks it), the
    plan stays correct in coverage, and its FLOPs are at least the rule's."""
    from gemm_tlr_gb300 import flops as fl
    n, b = 2048, 128
    nt = n // b
    ra = np.fromfunction(lambda i, k: np.where((k % 2) == 0, 8, 40), (nt, nt)).astype(np.int64)
    rb = np.fromfunction(lambda k, j: np.where((k % 2) == 0, 40, 8), (nt, nt)).astype(np.int64)
    rng = np.random.default_rng(8)
    A = ti.make_tlr(rng, n, b, None, "bf16", ranks=ra)
    B = ti.make_tlr(rng, n, b, None, "bf16", ranks=rb)
    p = ti.Problem("alternating", A, B, "N", "N", 1.0, 0.0, None, n, n, "bf16")
    Ad, Bd, keep, opA, opB = _fake(p)
    st, msg, info = g.tlr_debug_check_plan(opA, opB, Ad, Bd, 1 << 40, g.TLR_ORDER_TRIPLE)
    assert st == 0, msg
    rule = fl.executed_flops_triple(p)["total"]
    assert info["flops_executed"] >= rule
    assert info["flops_executed"] < fl.executed_flops(p, "R")["total"]


@pytest.mark.parametrize("make", [lambda: ti.problem(5, scale_down=4), lambda: ti.asym_grid(2048, 256),
                                  lambda: ti.asym_grid(4096, 256), lambda: ti.skewed_grid(4096, "bf16")],
                         ids=["cfg5/4", "asym2048", "asym4096", "skewed"])
def test_auto_order_follows_the_final_stage_costs(g, make):
    """tlr_analyze's per-triple final cost F_P equals the independent count, and
    AUTO takes the per-triple order exactly when F_P <= 0.9 min(F_R, F_L)."""
    from gemm_tlr_gb300 import flops as fl
    p = make()
    A, B, keep, opA, opB = _fake(p)
    n = len(p.A.rdims)
    out = g.tlr_analyze(opA, opB, A, B, n, n, n)
    trip = fl.executed_flops_triple(p)
    base = fl.executed_flops(p, "R")
    # on the terms of F_R and F_L: the final products of the low-rank triples and
    # of the k = j blocks (the dense-tile terms every order shares left out)
    assert out["F_P"] == pytest.approx(trip["stage3"], rel=1e-12)
    assert out["F_R"] == pytest.approx(base["stage3"], rel=1e-12)
    rects = g.tlr_debug_plan_rects(opA, opB, A, B, p.budget or (1 << 40), g.TLR_ORDER_AUTO)
    want = out["F_P"] <= 0.9 * min(out["F_R"], out["F_L"])
    assert ({r[4] for r in rects} == {"P"}) == want
    assert base["total"] > 0
