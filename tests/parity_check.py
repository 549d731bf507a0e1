"""Parity measures shared by the GPU tests: whole-block, per output tile, per region.

One relative Frobenius norm over all of C can hide a wrong output tile: a 10 %
error confined to one tile of a 16 x 16 grid moves the whole-C figure by about
10 % / 16. So every comparison also takes the largest relative error over the
output tiles of C (the b x b grid of op(A)'s rows by op(B)'s columns, boundary
tiles included), at the same tolerance, and products with a boundary tile are
also checked region by region: the interior, the boundary column C_12, the
boundary row C_21 and the corner C_22 ("TLR Matrix Multiplication", section
"Introduction: TLR GEMM", the four disjoint output regions).

A tile whose reference is zero (or nearly) is measured against a floor of
1e-3 x the root-mean-square tile norm, so it must stay near zero in absolute
terms instead of dividing by zero.
"""
from __future__ import annotations

import numpy as np


def rel(a, b) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def axis_groups(idx, b: int):
    """Positions of `idx` (indices along one axis of C) grouped by the b-wide tile they fall in."""
    groups = {}
    for pos, x in enumerate(np.asarray(idx)):
        groups.setdefault(int(x) // b, []).append(pos)
    return [np.array(v) for _, v in sorted(groups.items())]


def tile_errors(got, ref, row_idx, col_idx, b: int) -> np.ndarray:
    """Relative Frobenius error of every output tile (rows x cols of sampled or whole C).

    `row_idx` / `col_idx` are the indices into C of the rows / columns of
    `got` and `ref`; tiles are the b-wide blocks of C they fall in."""
    rg, cg = axis_groups(row_idx, b), axis_groups(col_idx, b)
    ntiles = len(rg) * len(cg)
    floor = 1e-3 * np.linalg.norm(ref) / np.sqrt(max(ntiles, 1))
    out = np.zeros((len(rg), len(cg)))
    for a, r in enumerate(rg):
        for c, cc in enumerate(cg):
            g, f = got[np.ix_(r, cc)], ref[np.ix_(r, cc)]
            out[a, c] = np.linalg.norm(g - f) / max(np.linalg.norm(f), floor, 1e-300)
    return out


def region_errors(got, ref, row_idx, col_idx, m_int: int, n_int: int) -> dict:
    """Relative error of each of the four regions of C split at interior extents m_int x n_int."""
    rows, cols = np.asarray(row_idx), np.asarray(col_idx)
    parts = {"interior": (rows < m_int, cols < n_int), "C_12": (rows < m_int, cols >= n_int),
             "C_21": (rows >= m_int, cols < n_int), "C_22": (rows >= m_int, cols >= n_int)}
    out = {}
    for name, (rm, cm) in parts.items():
        if rm.any() and cm.any():
            out[name] = rel(got[np.ix_(rm, cm)], ref[np.ix_(rm, cm)])
    return out


def check(got, ref, tol: float, b: int, row_idx=None, col_idx=None, regions=None, what: str = ""):
    """Whole-block, per-tile and (when `regions` = (m_int, n_int)) per-region checks at `tol`.

    Returns the measured errors; raises AssertionError naming the worst tile
    or region when any of them is above `tol`."""
    got = np.asarray(got)
    ref = np.asarray(ref)
    if row_idx is None:
        row_idx = np.arange(ref.shape[0])
    if col_idx is None:
        col_idx = np.arange(ref.shape[1])
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    whole = rel(got, ref)
    te = tile_errors(got, ref, row_idx, col_idx, b)
    worst = np.unravel_index(int(np.argmax(te)), te.shape)
    res = {"whole": whole, "tile_max": float(te.max()), "worst_tile": tuple(int(x) for x in worst)}
    assert whole <= tol, f"{what}: whole rel Frobenius {whole:.3e} > {tol}"
    assert te.max() <= tol, (f"{what}: output tile {res['worst_tile']} rel Frobenius {te.max():.3e} > {tol} "
                             f"(whole {whole:.3e})")
    if regions is not None:
        re = region_errors(got, ref, row_idx, col_idx, *regions)
        res["regions"] = re
        for name, e in re.items():
            assert e <= tol, f"{what}: region {name} rel Frobenius {e:.3e} > {tol}"
    return res


def interior_extents(p):
    """(m_int, n_int) of C when op(A) or op(B) has a boundary tile, else None."""
    b = p.A.b if p.A.kind == "tlr" else p.B.b
    if p.m % b == 0 and p.n % b == 0:
        return None
    return (p.m // b) * b, (p.n // b) * b


def tile_size(p) -> int:
    """Tile size of C's grid: the TLR operand's b."""
    return p.A.b if p.A.kind == "tlr" else p.B.b
