"""The parity checker itself (no GPU): a wrong output tile or region must fail it.

Mistakes are planted on the CPU in a copy of the oracle's own result, standing
in for a GPU output array, at sizes where the whole-C norm alone would still
pass.
"""
import numpy as np
import pytest

import tlr_inputs as ti
from parity_check import check, interior_extents, region_errors, tile_errors, tile_size


def _noisy(ref, rel_noise, seed=0):
    rng = np.random.default_rng(seed)
    return ref + rel_noise * np.abs(ref).mean() * rng.standard_normal(ref.shape)


def test_clean_result_passes_every_measure():
    rng = np.random.default_rng(1)
    ref = rng.standard_normal((512, 512))
    res = check(_noisy(ref, 1e-4), ref, 1e-2, 32)
    assert res["whole"] < 1e-3 and res["tile_max"] < 1e-3


def test_one_wrong_tile_fails_although_the_whole_norm_passes():
    rng = np.random.default_rng(2)
    ref = rng.standard_normal((512, 512))          # 16 x 16 tiles of 32
    got = _noisy(ref, 1e-4)
    got[96:128, 160:192] *= 1.05                   # tile (3, 5) off by 5 %
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2
    with pytest.raises(AssertionError, match=r"output tile \(3, 5\)"):
        check(got, ref, 1e-2, 32)


def test_wrong_tile_in_sampled_entries_is_found():
    rng = np.random.default_rng(3)
    n, b = 2048, 256
    rows = np.sort(rng.choice(n, 40, replace=False))
    cols = np.sort(rng.choice(n, 40, replace=False))
    ref = rng.standard_normal((rows.size, cols.size))
    got = _noisy(ref, 1e-4)
    r_in = (rows // b) == 6
    c_in = (cols // b) == 1
    got[np.ix_(r_in, c_in)] *= 1.04
    te = tile_errors(got, ref, rows, cols, b)
    assert te.max() > 0.03 and np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2
    with pytest.raises(AssertionError, match="output tile"):
        check(got, ref, 1e-2, b, rows, cols)


@pytest.mark.parametrize("region", ["interior", "C_12", "C_21", "C_22"])
def test_each_boundary_region_is_checked_on_its_own(region):
    rng = np.random.default_rng(4)
    m_int = n_int = 19 * 16
    n = m_int + 8                                  # 19 full tiles of 16 and an 8-wide boundary
    ref = rng.standard_normal((n, n))
    got = _noisy(ref, 1e-4)
    sl = {"interior": (slice(0, m_int), slice(0, n_int)), "C_12": (slice(0, m_int), slice(n_int, n)),
          "C_21": (slice(m_int, n), slice(0, n_int)), "C_22": (slice(m_int, n), slice(n_int, n))}[region]
    got[sl] *= 1.03
    re = region_errors(got, ref, np.arange(n), np.arange(n), m_int, n_int)
    assert re[region] > 2e-2 and all(v < 1e-3 for k, v in re.items() if k != region)
    with pytest.raises(AssertionError):
        check(got, ref, 2e-2, 10**6, regions=(m_int, n_int))   # tile check off (one tile): the region check alone


def test_planted_tile_error_on_an_oracle_result(oracle_lib):
    """The boundary workload at 1/8 size: the oracle's C with one output tile 3 % off
    passes the whole-C norm at the TF32 tolerance but not the per-tile check."""
    p = ti.problem(3, scale_down=8, zero_diag=True, beta_override=0.0)
    ref = oracle_lib.gemm_problem(p)
    b = tile_size(p)
    assert interior_extents(p) == ((p.m // b) * b, (p.n // b) * b)
    check(_noisy(ref, 1e-5), ref, 2e-3, b, regions=interior_extents(p))
    got = ref.copy()
    got[2 * b:3 * b, 7 * b:8 * b] *= 1.03
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 2e-3
    with pytest.raises(AssertionError, match=r"output tile \(2, 7\)"):
        check(got, ref, 2e-3, b, regions=interior_extents(p))
    corner = ref.copy()
    corner[-1, -1] += 0.5 * np.abs(ref).max()      # one entry of the boundary corner C_22
    with pytest.raises(AssertionError):
        check(corner, ref, 2e-3, b, regions=interior_extents(p))
