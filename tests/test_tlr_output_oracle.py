"""Pins of the TLR-output oracle (no GPU): closed forms, exact recovery, planted mistakes.

The oracle (oracle/tlr_output.py) compresses each off-diagonal tile of the dense
product to the smallest rank whose discarded singular values stay within eps of
the tile's Frobenius norm ("TLR Matrix Multiplication", section "Introduction:
TLR GEMM"; the recompression rule is this build's reading).
"""
import math

import numpy as np
import pytest

import tlr_inputs as ti
from oracle import tlr_output as to


def _orthogonal(rng, n):
    q, r = np.linalg.qr(rng.standard_normal((n, n)))
    return q * np.sign(np.diag(r))


def _spectrum_tile(rng, sigma):
    n = len(sigma)
    return _orthogonal(rng, n) @ np.diag(sigma) @ _orthogonal(rng, n).T


def _rule_rank(sigma, eps):
    """The truncation rule written out as a plain loop: smallest r with the
    discarded energy at most eps^2 of the total."""
    total = sum(s * s for s in sigma)
    for r in range(len(sigma) + 1):
        if sum(s * s for s in sigma[r:]) <= eps * eps * total:
            return r
    return len(sigma)


@pytest.mark.parametrize("eps", [0.3, 1e-1, 1e-2, 1e-3, 1e-6])
def test_prescribed_spectrum_closed_form(eps):
    """A tile with singular values 2^-s: the rank is the rule's and the error is
    exactly sqrt(sum of the discarded sigma^2) / ||sigma|| (Eckart-Young)."""
    rng = np.random.default_rng(1)
    sigma = [2.0 ** -s for s in range(40)]
    tile = _spectrum_tile(rng, sigma)
    U, V, r, err = to.compress_tile(tile, eps, 40)
    want_r = _rule_rank(sigma, eps)
    assert r == want_r
    want_err = math.sqrt(sum(s * s for s in sigma[r:])) / math.sqrt(sum(s * s for s in sigma))
    assert err == pytest.approx(want_err, rel=1e-9, abs=1e-15)
    got = np.linalg.norm(tile - U @ V.T) / np.linalg.norm(tile)
    assert got == pytest.approx(want_err, rel=1e-6, abs=1e-13)
    assert got <= eps * (1 + 1e-12)
    assert U.shape == (40, r) and V.shape == (40, r)


def test_rank_cap_keeps_r_max_and_reports_the_larger_error():
    rng = np.random.default_rng(2)
    sigma = [1.0 / (1 + s) for s in range(32)]
    tile = _spectrum_tile(rng, sigma)
    U, V, r, err = to.compress_tile(tile, 1e-4, 5)
    assert r == 5
    assert err == pytest.approx(math.sqrt(sum(s * s for s in sigma[5:]) / sum(s * s for s in sigma)), rel=1e-9)
    assert err > 1e-4


def _identity_like(rng, n, b):
    """A TLR matrix equal to the identity: dense identity diagonal tiles, every
    off-diagonal tile of rank 0."""
    nt = n // b
    I = ti.make_tlr(rng, n, b, None, "f32", ranks=np.zeros((nt, nt), dtype=np.int64))
    for t in range(nt):
        I.D[t * b * b:(t + 1) * b * b] = np.eye(b, dtype=np.float32).reshape(-1, order="F")
    return I


def test_product_with_identity_recovers_the_operand_ranks():
    """C = A I: every off-diagonal tile of C is A's tile U_ik V_ik^T, whose rank
    (random factors) is exactly r_ik, and the diagonal stays dense."""
    rng = np.random.default_rng(3)
    n, b = 384, 64
    A = ti.make_tlr(rng, n, b, ti.rank_uniform(0, 12), "f32")
    I = _identity_like(rng, n, b)
    p = ti.Problem("times_identity", A, I, "N", "N", 1.0, 0.0, None, n, n, "f32")
    out = to.tlr_output_product(p, 1e-10, b)
    nt = n // b
    for i in range(nt):
        for j in range(nt):
            if i != j:
                assert out["ranks"][i, j] == A.ranks[i, j], (i, j)
    assert out["dense_diagonal"]
    import oracle
    dense = oracle.gemm_problem(p)
    assert np.linalg.norm(to.expand(out) - dense) <= 1e-9 * np.linalg.norm(dense)


def test_beta_term_is_part_of_the_compressed_tile():
    """alpha op(A) op(B) + beta C0 is compressed as one tile: with A I and a C0
    whose tiles are rank-one outer products (stored in fp32, so below 1e-6 they
    are full rank), every off-diagonal tile of the result has rank r_ik + 1."""
    rng = np.random.default_rng(4)
    n, b = 256, 64
    A = ti.make_tlr(rng, n, b, ti.rank_uniform(1, 8), "f32")
    I = _identity_like(rng, n, b)
    x = rng.standard_normal(n)
    y = rng.standard_normal(n)
    C0 = np.outer(x, y).astype(np.float32).reshape(-1, order="F")
    p = ti.Problem("a_plus_rank_one", A, I, "N", "N", 1.0, 0.5, C0, n, n, "f32")
    out = to.tlr_output_product(p, 1e-5, b)
    nt = n // b
    for i in range(nt):
        for j in range(nt):
            if i != j:
                assert out["ranks"][i, j] == A.ranks[i, j] + 1, (i, j)
    without = to.tlr_output_product(ti.Problem("a", A, I, "N", "N", 1.0, 0.0, None, n, n, "f32"), 1e-5, b)
    assert (without["ranks"] == np.where(np.eye(nt, dtype=bool), 0, A.ranks)).all()


def test_planted_mistakes_fail_the_pins():
    """An off-by-one truncation breaks the error bound; swapped factors break the
    recovery of the operand."""
    rng = np.random.default_rng(5)
    sigma = [2.0 ** -s for s in range(40)]
    tile = _spectrum_tile(rng, sigma)
    eps = 1e-3
    U, V, r, _ = to.compress_tile(tile, eps, 40)
    short = np.linalg.norm(tile - U[:, :r - 1] @ V[:, :r - 1].T) / np.linalg.norm(tile)
    assert short > eps                                    # one rank fewer misses the bound
    assert np.linalg.norm(tile - V @ U.T) > 0.5 * np.linalg.norm(tile)   # factors swapped
