"""GPU parity for fp16 operands and for the pages' skewed-rank 8 x 8 workload.

fp16 keeps 10 stored mantissa bits against bf16's 7, so its rounding errors are 8x
smaller; the products keep fp32 accumulation and an fp16 S, T and P. The
tolerance below is the bf16 bound (1e-2) scaled by that ratio with a 2x margin
(2.5e-3). The skewed workload runs in fp32 (TF32), bf16 and fp16, at sizes the
oracle computes whole and, for fp16, at the pages' largest size on sampled
entries.
"""
import numpy as np
import pytest

import tlr_inputs as ti
from parity_check import check, interior_extents, tile_size
from test_parity_gpu import TOL as _TOL, handle, rel, run, sample_indices, torch_cuda  # noqa: F401

pytestmark = pytest.mark.gpu
TOL = dict(_TOL, f16=2.5e-3)


def check_p(out, ref, p, rows=None, cols=None):
    """Whole, per-tile and per-region parity at this element type's tolerance."""
    return check(out, ref, TOL[p.dtype], tile_size(p), rows, cols, regions=interior_extents(p), what=p.name)


@pytest.mark.parametrize("cfg,scale", [(4, 8), (4, 4), (5, 8), (5, 4)])
@pytest.mark.parametrize("variant", ["whole", "lowrank_only", "dense_only"])
def test_fp16_workloads_match_oracle(oracle_lib, handle, cfg, scale, variant):
    kw = {}
    if variant == "lowrank_only":
        kw = dict(zero_diag=True, beta_override=0.0)
    elif variant == "dense_only":
        kw = dict(zero_lowrank=True)
    p = ti.problem(cfg, scale_down=scale, dtype_override="f16", **kw)
    out, info = run(p, handle)
    res = check_p(out, oracle_lib.gemm_problem(p), p)
    print(f"{p.name} {variant}: {res}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n", [2048, 4096])
def test_skewed_grid_matches_oracle(oracle_lib, handle, dtype, n):
    p = ti.skewed_grid(n, dtype)
    out, info = run(p, handle)
    res = check_p(out, oracle_lib.gemm_problem(p), p)
    print(f"{p.name}: {res}")


@pytest.mark.parametrize("n", [65536])
def test_skewed_grid_largest_fp16_sampled(oracle_lib, handle, n):
    """The pages' largest fp16 case (N = 65536, b = 8192) on sampled rows and columns of every tile."""
    p = ti.skewed_grid(n, "f16")
    out_rows = sample_indices(p.m, p.A.b, seed=1)
    out_cols = sample_indices(p.n, p.A.b, seed=2)
    import gemm_tlr_gb300 as g
    from gemm_tlr_gb300.device import DeviceProblem
    dp = DeviceProblem(p)
    try:
        dp.make_plan(handle)
        dp.run()
        assert g.tlr_get_device_status(handle) == 0
        import torch
        Cd = dp.C.view(p.n, p.m)                          # column-major: Cd[col, row]
        sub = Cd[torch.as_tensor(out_cols, device=Cd.device)][:, torch.as_tensor(out_rows, device=Cd.device)]
        got = sub.double().cpu().numpy().T
    finally:
        dp.close()
    res = check_p(got, oracle_lib.gemm_problem(p, out_rows, out_cols), p, out_rows, out_cols)
    print(f"{p.name} sampled: {res}")


@pytest.mark.parametrize("opA,opB", [("N", "N"), ("N", "T"), ("T", "N"), ("T", "T")])
def test_fp16_transposes_with_boundary(oracle_lib, handle, opA, opB):
    """fp16 through every operand orientation, with a 72-wide boundary tile and beta != 0."""
    rng = np.random.default_rng(31)
    N, b = 456, 128
    A = ti.make_tlr(rng, N, b, ti.rank_uniform(0, 40), "f16")
    B = ti.make_tlr(rng, N, b, ti.rank_uniform(0, 40), "f16")
    C = rng.standard_normal(N * N).astype(np.float32)
    p = ti.Problem("transpose_f16", A, B, opA, opB, 0.75, -1.25, C, N, N, "f16")
    out, _ = run(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)


@pytest.mark.parametrize("left_dense", [True, False])
def test_fp16_dense_operand(oracle_lib, handle, left_dense):
    """A dense fp16 operand on either side of a TLR one (96-wide tiles, 72-wide boundary)."""
    rng = np.random.default_rng(32)
    if left_dense:
        A = ti.make_dense(rng, 320, 456, "f16")
        B = ti.make_tlr(rng, 456, 96, ti.rank_uniform(1, 48), "f16")
        m, n = 320, 456
    else:
        A = ti.make_tlr(rng, 456, 96, ti.rank_uniform(1, 48), "f16")
        B = ti.make_dense(rng, 456, 256, "f16")
        m, n = 456, 256
    p = ti.Problem("dense_tlr_f16", A, B, "N", "N", 1.0, 0.0, None, m, n, "f16")
    out, _ = run(p, handle)
    check_p(out, oracle_lib.gemm_problem(p), p)
