"""Seeded synthetic inputs for Tile-Low-Rank GEMM.

This module only *draws and lays out* inputs. It holds none of the product's
arithmetic: no factor products, no tile reconstruction, no GEMM. Both the CPU
oracle (under ``oracle/``) and the GPU path (``gemm_tlr_gb300``) consume what it
returns, and neither imports the other.

Storage convention (the TLR format of "Tile-Low-Rank GEMM: Designing Storage
Around the Contraction", section "Packing for the contraction", and "TLR Matrix
Multiplication", section "Introduction: TLR GEMM"):

* A TLR matrix is a grid of tiles. Tile row ``i`` has ``d_i`` rows and tile
  column ``k`` has ``d_k`` columns; all interior tiles are ``b x b``; when the
  order ``N`` is not a multiple of ``b`` the last tile row/column has
  ``b_rem = N - m*b`` rows/columns (``m = N // b``).
* With ``diag_dense`` the diagonal tiles are dense; every other tile ``(i,k)``
  is ``U_ik V_ik^T`` with its own rank ``r_ik`` (0 allowed).
* Outer factors ``U`` are packed by tile row (row ``i`` ascending, then ``k``
  ascending, dense tiles skipped); inner factors ``V`` are packed by tile column
  (column ``k`` ascending, then ``i`` ascending). Every factor is column-major
  with leading dimension equal to its own dense dimension, and occupies exactly
  ``r_ik`` columns (no padding).
* Boundary panels (same page 2, "Introduction"): the interior ``m x m`` grid is
  stored in ``U``/``V``/``D``; the boundary column ``u`` (tiles ``(i, m)``),
  the boundary row ``v^T`` (tiles ``(m, j)``) and the dense corner ``gamma``
  have buffers of their own: ``bu_U``/``bu_V`` hold the outer/inner factors of
  the boundary column packed by ascending ``i``, ``bv_U``/``bv_V`` those of the
  boundary row packed by ascending ``j``.

All arrays are float32 numpy arrays. For bf16 and fp16 inputs the values are
rounded to that type (round-to-nearest-even) and kept as float32 holding exact
values of it; ``bf16_bits`` turns bf16 values into the 16-bit payload for upload.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Dict, Optional, Tuple

import numpy as np

__all__ = [
    "var_rank_grid", "bf16_round", "f16_round", "bf16_bits", "TLRMatrix", "DenseMatrix", "Problem",
    "make_tlr", "make_dense", "problem", "CONFIG_NAMES", "tile_dims",
    "rank_fixed", "rank_uniform", "rank_inverse_distance", "rank_exp_decay", "rank_skewed",
    "skewed_grid", "asym_grid", "rank_split_rows",
]


# ---------------------------------------------------------------- dtype helpers
def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def f16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest fp16 (ties to even); returns float32."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """16-bit payload of bf16-exact float32 values (upper half of the word)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def tile_dims(n: int, b: int) -> list:
    """Dense dimension of every tile along one axis of order ``n``."""
    m, rem = divmod(n, b)
    return [b] * m + ([rem] if rem else [])


# ---------------------------------------------------------------- containers
@dataclass
class TLRMatrix:
    rows: int
    cols: int
    b: int
    diag_dense: bool
    ranks: np.ndarray              # (nt_r, nt_c) int32, dense tiles hold 0
    dtype: str                     # "f32", "bf16" or "f16"
    U: np.ndarray
    V: np.ndarray
    D: Optional[np.ndarray] = None         # b*b*m, tile i at i*b*b
    bu_U: Optional[np.ndarray] = None
    bu_V: Optional[np.ndarray] = None
    bv_U: Optional[np.ndarray] = None
    bv_V: Optional[np.ndarray] = None
    gamma: Optional[np.ndarray] = None
    # Per-tile views into the buffers above, filled by the packer itself:
    # (i,k) -> ("lr", U_ik (d_i x r), V_ik (d_k x r)) or ("dense", D_ii).
    tiles: Optional[Dict[Tuple[int, int], tuple]] = None

    @property
    def kind(self) -> str:
        return "tlr"

    @property
    def rdims(self):
        return tile_dims(self.rows, self.b)

    @property
    def cdims(self):
        return tile_dims(self.cols, self.b)

    def nbytes_device(self) -> int:
        es = 4 if self.dtype == "f32" else 2
        n = 0
        for a in (self.U, self.V, self.D, self.bu_U, self.bu_V, self.bv_U, self.bv_V, self.gamma):
            if a is not None:
                n += a.size * es
        return n


@dataclass
class DenseMatrix:
    rows: int
    cols: int
    dtype: str
    data: np.ndarray               # column-major, ld = rows, flattened float32

    @property
    def kind(self) -> str:
        return "dense"


@dataclass
class Problem:
    name: str
    A: object
    B: object
    opA: str                       # "N" or "T"
    opB: str
    alpha: float
    beta: float
    C: Optional[np.ndarray]        # column-major flattened float32, or None (beta == 0)
    m: int                         # rows of C
    n: int                         # cols of C
    dtype: str
    budget: Optional[int] = None   # workspace budget in bytes (None: unlimited)
    note: str = ""
    extra: dict = field(default_factory=dict)


# ---------------------------------------------------------------- rank rules
def rank_fixed(r: int) -> Callable:
    def f(rng, nt_r, nt_c, rd, cd):
        return np.full((nt_r, nt_c), r, dtype=np.int64)
    return f


def rank_uniform(lo: int, hi: int) -> Callable:
    """Independent integer ranks, uniform on [lo, hi] inclusive."""
    def f(rng, nt_r, nt_c, rd, cd):
        return rng.integers(lo, hi + 1, size=(nt_r, nt_c), dtype=np.int64)
    return f


def rank_skewed(lo: int, hi: int) -> Callable:
    """Independent ranks on [lo, hi], skewed towards lo: lo + floor((hi - lo + 1) u^2), u ~ U[0, 1).

    The pages give only the interval and the word "skewed"; squaring a uniform
    draw is the reading taken here (density falling linearly in sqrt, mean
    lo + (hi - lo + 1) / 3).
    """
    def f(rng, nt_r, nt_c, rd, cd):
        u = rng.random(size=(nt_r, nt_c))
        return np.minimum(hi, lo + np.floor((hi - lo + 1) * u * u).astype(np.int64))
    return f


def _round_half_up(x: float) -> int:
    return int(math.floor(x + 0.5))


def rank_inverse_distance(num: float, floor_: int) -> Callable:
    """r_ij = max(floor_, round(num / (1 + |i-j|)))."""
    def f(rng, nt_r, nt_c, rd, cd):
        r = np.zeros((nt_r, nt_c), dtype=np.int64)
        for i in range(nt_r):
            for j in range(nt_c):
                r[i, j] = max(floor_, _round_half_up(num / (1 + abs(i - j))))
        return r
    return f


def rank_exp_decay(scale: float, length: float, lo: int, hi: int) -> Callable:
    """r_ij = clamp(round(scale * exp(-|i-j| / length)), lo, hi)."""
    def f(rng, nt_r, nt_c, rd, cd):
        r = np.zeros((nt_r, nt_c), dtype=np.int64)
        for i in range(nt_r):
            for j in range(nt_c):
                r[i, j] = min(hi, max(lo, _round_half_up(scale * math.exp(-abs(i - j) / length))))
        return r
    return f


# ---------------------------------------------------------------- generators
def _draw(rng, n: int, scale: float, dtype: str) -> np.ndarray:
    a = rng.standard_normal(n, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    if dtype == "bf16":
        a = bf16_round(a)
    elif dtype == "f16":
        a = f16_round(a)
    return a


def make_tlr(rng, n: int, b: int, rank_rule: Callable, dtype: str, *,
             factor_scale: Optional[float] = None, diag_scale: float = 1.0,
             diag_dense: bool = True, cols: Optional[int] = None,
             ranks: Optional[np.ndarray] = None, keep_tiles: bool = False) -> TLRMatrix:
    """Draw one TLR matrix.

    Draw order: ranks (unless given), then the interior ``U`` buffer, ``V``
    buffer, ``D`` buffer, then the boundary buffers ``bu_U``, ``bu_V``,
    ``bv_U``, ``bv_V``, ``gamma``. Factors ~ N(0,1) * factor_scale (default
    1/sqrt(b)), dense tiles ~ N(0,1) * diag_scale.
    """
    rows = n
    cols = n if cols is None else cols
    rd, cd = tile_dims(rows, b), tile_dims(cols, b)
    ntr, ntc = len(rd), len(cd)
    if diag_dense and rows != cols:
        raise ValueError("dense diagonal needs a square matrix")
    boundary = (rows % b) != 0 or (cols % b) != 0
    if boundary and not (diag_dense and rows == cols):
        raise ValueError("boundary panels are defined for square matrices with a dense diagonal")
    if ranks is None:
        ranks = rank_rule(rng, ntr, ntc, rd, cd)
    ranks = np.array(ranks, dtype=np.int64)
    for i in range(ntr):
        for k in range(ntc):
            if diag_dense and i == k:
                ranks[i, k] = 0
            else:
                ranks[i, k] = max(0, min(int(ranks[i, k]), rd[i], cd[k]))
    ranks = ranks.astype(np.int32)
    fs = (1.0 / math.sqrt(b)) if factor_scale is None else factor_scale
    m = rows // b if boundary else ntr          # interior tile count (square case)
    mr = m if boundary else ntr
    mc = m if boundary else ntc

    def lowrank(i, k):
        return not (diag_dense and i == k)

    # interior sizes (columns of the packed buffers)
    u_cols = sum(int(ranks[i, k]) for i in range(mr) for k in range(mc) if lowrank(i, k))
    U = _draw(rng, b * u_cols, fs, dtype)
    V = _draw(rng, b * u_cols, fs, dtype)
    D = _draw(rng, b * b * mr, diag_scale, dtype) if diag_dense and mr > 0 else None
    bu_U = bu_V = bv_U = bv_V = gamma = None
    brem = rows - m * b
    if boundary:
        cu = sum(int(ranks[i, m]) for i in range(m))
        cv = sum(int(ranks[m, j]) for j in range(m))
        bu_U = _draw(rng, b * cu, fs, dtype)
        bu_V = _draw(rng, brem * cu, fs, dtype)
        bv_U = _draw(rng, brem * cv, fs, dtype)
        bv_V = _draw(rng, b * cv, fs, dtype)
        gamma = _draw(rng, brem * brem, diag_scale, dtype)

    tiles = None
    if keep_tiles:
        tiles = {}
        # interior U: row-major tile order
        col = 0
        uoff = {}
        for i in range(mr):
            for k in range(mc):
                if lowrank(i, k):
                    uoff[(i, k)] = col
                    col += int(ranks[i, k])
        col = 0
        voff = {}
        for k in range(mc):
            for i in range(mr):
                if lowrank(i, k):
                    voff[(i, k)] = col
                    col += int(ranks[i, k])
        for i in range(mr):
            for k in range(mc):
                if not lowrank(i, k):
                    tiles[(i, k)] = ("dense", D[i * b * b:(i + 1) * b * b].reshape(b, b, order="F"))
                    continue
                r = int(ranks[i, k])
                Ui = U[b * uoff[(i, k)]: b * (uoff[(i, k)] + r)].reshape(b, r, order="F")
                Vi = V[b * voff[(i, k)]: b * (voff[(i, k)] + r)].reshape(b, r, order="F")
                tiles[(i, k)] = ("lr", Ui, Vi)
        if boundary:
            c = 0
            for i in range(m):
                r = int(ranks[i, m])
                tiles[(i, m)] = ("lr", bu_U[b * c: b * (c + r)].reshape(b, r, order="F"),
                                 bu_V[brem * c: brem * (c + r)].reshape(brem, r, order="F"))
                c += r
            c = 0
            for j in range(m):
                r = int(ranks[m, j])
                tiles[(m, j)] = ("lr", bv_U[brem * c: brem * (c + r)].reshape(brem, r, order="F"),
                                 bv_V[b * c: b * (c + r)].reshape(b, r, order="F"))
                c += r
            tiles[(m, m)] = ("dense", gamma.reshape(brem, brem, order="F"))
    return TLRMatrix(rows=rows, cols=cols, b=b, diag_dense=diag_dense, ranks=ranks,
                     dtype=dtype, U=U, V=V, D=D, bu_U=bu_U, bu_V=bu_V, bv_U=bv_U,
                     bv_V=bv_V, gamma=gamma, tiles=tiles)


def make_dense(rng, rows: int, cols: int, dtype: str, scale: float = 1.0) -> DenseMatrix:
    return DenseMatrix(rows=rows, cols=cols, dtype=dtype, data=_draw(rng, rows * cols, scale, dtype))


# ---------------------------------------------------------------- workloads
CONFIG_NAMES = {
    1: "tiny_fixed_rank_f32_N512_b64",
    2: "var_rank_f32_N4096_b256",
    3: "boundary_TN_f32_N10000_b512",
    4: "one_tlr_bf16_16384x16384_b1024_x_16384x4096",
    5: "large_var_rank_bf16_N32768_b1024",
}


def var_rank_grid(n: int, *, b: int = 1024, dtype: str = "bf16", seed: int = 0,
                  budget: Optional[int] = None) -> Problem:
    """The large variable-rank family at another order: b = 1024 tiles with the
    same rank rule, clamp(round(256 exp(-|i-j|/4)), 8, 256), so every tile has
    the large product's shape and only the grid (n / b tiles a side) changes.
    A budget of 2 GiB scaled by (n / 32768)^2 unless given.
    """
    if n % b:
        raise ValueError("n must be a multiple of b")
    rng = np.random.default_rng(seed)
    rule = rank_exp_decay(256, 4.0, 8, 256)
    A = make_tlr(rng, n, b, rule, dtype)
    Bm = make_tlr(rng, n, b, rule, dtype)
    if budget is None:
        budget = int((2 << 30) * (n / 32768) ** 2)
    return Problem(f"var_rank_{dtype}_N{n}_b{b}", A, Bm, "N", "N", 1.0, 0.0, None, n, n, dtype, budget=budget)


def skewed_grid(n: int, dtype: str, *, seed: int = 0, keep_tiles: bool = False, budget: Optional[int] = None) -> Problem:
    """The pages' variable-rank workload: dense C <- TLR x TLR on an 8 x 8 tile
    grid, b = n / 8, every off-diagonal tile with its own rank drawn from a
    skewed distribution on [b/32, b/16] ("Tile-Low-Rank GEMM: Designing Storage
    Around the Contraction", section "Results"), dense diagonal tiles, factors
    ~N(0,1)/sqrt(b), dense tiles ~N(0,1), alpha = 1, beta = 0.
    """
    if n % 8 or (n // 8) % 32:
        raise ValueError("n must be a multiple of 256")
    rng = np.random.default_rng(seed)
    b = n // 8
    rule = rank_skewed(b // 32, b // 16)
    A = make_tlr(rng, n, b, rule, dtype, keep_tiles=keep_tiles)
    Bm = make_tlr(rng, n, b, rule, dtype, keep_tiles=keep_tiles)
    return Problem(f"skewed_8x8_{dtype}_N{n}", A, Bm, "N", "N", 1.0, 0.0, None, n, n, dtype, budget=budget)


def rank_split_rows(hi: int, scale: float, length: float, lo: int) -> Callable:
    """Tile rows in the upper half at rank `hi` everywhere; the lower half
    r_ik = clamp(round(scale exp(-|i-k| / length)), lo, hi)."""
    def f(rng, nt_r, nt_c, rd, cd):
        r = np.zeros((nt_r, nt_c), dtype=np.int64)
        for i in range(nt_r):
            for k in range(nt_c):
                r[i, k] = hi if 2 * i < nt_r else min(hi, max(lo, _round_half_up(scale * math.exp(-abs(i - k) / length))))
        return r
    return f


def asym_grid(n: int, b: int, dtype: str = "bf16", *, seed: int = 0, budget: Optional[int] = None) -> Problem:
    """TLR x TLR with unlike rank maps, so that the right, left, per-rectangle and
    per-triple orders all execute different FLOP counts: A's upper tile rows all
    have rank b/4 and its lower ones decay away from the diagonal,
    clamp(round(b/8 exp(-|i-k|/2)), 2, b/4); B's ranks are uniform on [b/32, b/8]
    per tile. Factors ~N(0,1)/sqrt(b), dense diagonal tiles ~N(0,1), alpha = 1,
    beta = 0 (a test and measurement workload, not one of the five)."""
    if n % b:
        raise ValueError("n must be a multiple of b")
    rng = np.random.default_rng(seed)
    A = make_tlr(rng, n, b, rank_split_rows(b // 4, b / 8, 2.0, 2), dtype)
    Bm = make_tlr(rng, n, b, rank_uniform(max(1, b // 32), b // 8), dtype)
    return Problem(f"asym_{dtype}_N{n}_b{b}", A, Bm, "N", "N", 1.0, 0.0, None, n, n, dtype, budget=budget)


def problem(cfg, *, seed: int = 0, keep_tiles: bool = False, scale_down: int = 1,
            zero_diag: bool = False, zero_lowrank: bool = False, beta_override=None,
            alpha_override=None, dtype_override: Optional[str] = None) -> Problem:
    """Build one of the five graded workloads (or a smaller member of its family).

    ``cfg`` is 1..5. ``scale_down`` > 1 divides N (and for config 4 the dense
    width) while keeping the structure (tile grid shape, rank rule, boundary
    remainder ratio) so the oracle can run the whole product. ``zero_diag`` and
    ``zero_lowrank`` build the term-isolated variants (dense tiles, or every
    low-rank factor, replaced by zeros after drawing, so that the other values
    are the same seeded draws). ``dtype_override`` ("f16" for the bf16
    workloads) draws the same distributions rounded to another 16-bit type.
    """
    rng = np.random.default_rng(seed)
    kt = keep_tiles
    if cfg == 1:
        N, b = 512 // scale_down, 64 // scale_down
        A = make_tlr(rng, N, b, rank_fixed(8), "f32", keep_tiles=kt)
        Bm = make_tlr(rng, N, b, rank_fixed(8), "f32", keep_tiles=kt)
        p = Problem(CONFIG_NAMES[1], A, Bm, "N", "N", 1.0, 0.0, None, N, N, "f32")
    elif cfg == 2:
        N, b = 4096 // scale_down, 256 // scale_down
        lo, hi = (8, 64) if scale_down == 1 else (max(1, 8 // scale_down), max(2, 64 // scale_down))
        A = make_tlr(rng, N, b, rank_uniform(lo, hi), "f32", keep_tiles=kt)
        Bm = make_tlr(rng, N, b, rank_uniform(lo, hi), "f32", keep_tiles=kt)
        C = rng.standard_normal(N * N, dtype=np.float32)
        p = Problem(CONFIG_NAMES[2], A, Bm, "N", "N", 1.5, 0.5, C, N, N, "f32")
    elif cfg == 3:
        # 19 full tiles plus a ragged boundary tile of 272/512 of a tile.
        b = 512 // scale_down
        brem = 272 // scale_down
        brem += (-brem) % 4                      # keep 16-byte aligned fp32 columns
        N = 19 * b + brem
        num, fl = (128.0, 4) if scale_down == 1 else (128.0 / scale_down, 1)
        A = make_tlr(rng, N, b, rank_inverse_distance(num, fl), "f32", keep_tiles=kt)
        Bm = make_tlr(rng, N, b, rank_inverse_distance(num, fl), "f32", keep_tiles=kt)
        C = rng.standard_normal(N * N, dtype=np.float32)
        p = Problem(CONFIG_NAMES[3], A, Bm, "T", "N", 1.0, 1.0, C, N, N, "f32")
    elif cfg == 4:
        N, b, W = 16384 // scale_down, 1024 // scale_down, 4096 // scale_down
        lo, hi = (16, 256) if scale_down == 1 else (max(1, 16 // scale_down), max(2, 256 // scale_down))
        dt = dtype_override or "bf16"
        A = make_tlr(rng, N, b, rank_uniform(lo, hi), dt, keep_tiles=kt)
        Bm = make_dense(rng, N, W, dt)
        p = Problem(CONFIG_NAMES[4], A, Bm, "N", "N", 1.0, 0.0, None, N, W, dt)
    elif cfg == 5:
        N, b = 32768 // scale_down, 1024 // scale_down
        rule = rank_exp_decay(256 / scale_down, 4.0, max(1, 8 // scale_down), 256 // scale_down)
        dt = dtype_override or "bf16"
        A = make_tlr(rng, N, b, rule, dt, keep_tiles=kt)
        Bm = make_tlr(rng, N, b, rule, dt, keep_tiles=kt)
        budget = (2 << 30) // (scale_down * scale_down)
        p = Problem(CONFIG_NAMES[5], A, Bm, "N", "N", 1.0, 0.0, None, N, N, dt, budget=budget)
    else:
        raise ValueError(f"unknown config {cfg}")
    if dtype_override is not None and cfg in (1, 2, 3):
        raise ValueError("dtype_override applies to the 16-bit workloads (4, 5)")
    if dtype_override is not None:
        p.name = p.name.replace("bf16", dtype_override)
    if scale_down != 1:
        p.name += f"/scale{scale_down}"
    if zero_diag or zero_lowrank:
        for X in (p.A, p.B):
            _zero_parts(X, zero_diag, zero_lowrank)
        p.name += "/zero_diag" if zero_diag else "/zero_lowrank"
    if beta_override is not None:
        p.beta = beta_override
        if p.beta == 0.0:
            p.C = None
        elif p.C is None:
            p.C = np.random.default_rng(seed + 1).standard_normal(p.m * p.n, dtype=np.float32)
    if alpha_override is not None:
        p.alpha = alpha_override
    return p


def _zero_parts(X, zero_diag: bool, zero_lowrank: bool) -> None:
    if isinstance(X, DenseMatrix):
        return
    if zero_diag:
        for a in (X.D, X.gamma):
            if a is not None:
                a[:] = 0
    if zero_lowrank:
        for a in (X.U, X.V, X.bu_U, X.bu_V, X.bv_U, X.bv_V):
            if a is not None:
                a[:] = 0


def sketch(b: int, s: int, seed: int = 0) -> np.ndarray:
    """The random test matrix Omega (b x s, entries N(0, 1), float32) that the
    GPU recompression of TLR-output products takes as an input; the oracle's
    recompression is exact and draws nothing."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x5EC, b, s]))
    return rng.standard_normal((b, s)).astype(np.float32)
