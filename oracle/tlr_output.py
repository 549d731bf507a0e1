"""CPU fp64 oracle of the TLR-output product (test infrastructure).

"TLR Matrix Multiplication", section "Introduction: TLR GEMM", says only that the
TLR-output cases extend the dense-output product; "Tile-Low-Rank GEMM: Designing
Storage Around the Contraction", section "Many small GEMMs", says that TLR
compresses each tile of a regular grid independently, its rank following the
tile's local compressibility. Neither page describes the recompression. The
reading taken here, the plainest the text supports:

* the output keeps the tile grid of the product: op(A)'s row tiles by op(B)'s
  column tiles;
* for a square output whose operands both have dense diagonal tiles, the
  diagonal tiles of C stay dense;
* every other tile is the dense tile ``alpha (op(A) op(B))_ij + beta C0_ij``
  compressed to its truncated singular value decomposition with the smallest
  rank r for which the discarded part satisfies
  ``sqrt(sum_{s > r} sigma_s^2) <= eps * ||tile||_F`` (relative Frobenius
  error per tile; by Eckart and Young no rank-r factorisation does better),
  capped at ``r_max``; a tile whose tolerance needs more than ``r_max`` keeps
  ``r_max`` and reports its larger error;
* the factors are ``U = U_r diag(sigma_r)`` and ``V = V_r`` (the split of the
  singular values between the two factors is not fixed by the pages; only the
  product ``U V^T`` is compared).

The dense tiles come from the plain definition in ``tlr_oracle.c``; the SVD is
numpy's (LAPACK), in fp64. Pinned in ``tests/test_tlr_output_oracle.py`` by a
closed form (a tile with prescribed singular values), by the exact recovery of
an operand (a product with an identity factor), and by planted mistakes.
"""
from __future__ import annotations

import numpy as np


def truncation_rank(sigma: np.ndarray, eps: float, r_max: int) -> int:
    """Smallest r with sqrt(sum_{s >= r} sigma_s^2) <= eps * ||sigma||_2, at most r_max."""
    sigma = np.asarray(sigma, dtype=np.float64)
    total = float(np.sqrt(np.sum(sigma * sigma)))
    # tail[r] = sqrt(sum_{s >= r} sigma_s^2) for r = 0..n
    tail = np.sqrt(np.concatenate([np.cumsum((sigma * sigma)[::-1])[::-1], [0.0]]))
    r = int(np.argmax(tail <= eps * total)) if total > 0 else 0
    return min(r, int(r_max))


def compress_tile(tile: np.ndarray, eps: float, r_max: int):
    """(U, V, r, relative error) of one tile: U V^T is its truncated SVD."""
    tile = np.asarray(tile, dtype=np.float64)
    u, s, vt = np.linalg.svd(tile, full_matrices=False)
    r = truncation_rank(s, eps, r_max)
    norm = float(np.linalg.norm(s))
    err = float(np.sqrt(np.sum(s[r:] ** 2)) / norm) if norm > 0 else 0.0
    return u[:, :r] * s[:r], vt[:r, :].T.copy(), r, err


def tlr_output_product(p, eps: float, r_max: int) -> dict:
    """The TLR form of alpha op(A) op(B) + beta C0 for a problem ``p`` of ``tlr_inputs``.

    Returns ``{"ranks": (nI, nJ) int array (0 on dense tiles), "tiles": {(i, j):
    ("lr", U, V) | ("dense", D)}, "errors": (nI, nJ) relative errors, "rdims",
    "cdims", "dense_diagonal"}``.
    """
    import oracle
    C = oracle.gemm_problem(p)
    b = p.A.b if p.A.kind == "tlr" else p.B.b
    rd = [min(b, p.m - s) for s in range(0, p.m, b)]
    cd = [min(b, p.n - s) for s in range(0, p.n, b)]
    dense_diag = (p.m == p.n and p.A.kind == "tlr" and p.B.kind == "tlr" and p.A.diag_dense and p.B.diag_dense)
    ranks = np.zeros((len(rd), len(cd)), dtype=np.int64)
    errors = np.zeros((len(rd), len(cd)))
    tiles = {}
    r0 = 0
    for i, di in enumerate(rd):
        c0 = 0
        for j, dj in enumerate(cd):
            t = C[r0:r0 + di, c0:c0 + dj]
            if dense_diag and i == j:
                tiles[(i, j)] = ("dense", t.copy())
            else:
                U, V, r, err = compress_tile(t, eps, min(r_max, di, dj))
                tiles[(i, j)] = ("lr", U, V)
                ranks[i, j] = r
                errors[i, j] = err
            c0 += dj
        r0 += di
    return {"ranks": ranks, "tiles": tiles, "errors": errors, "rdims": rd, "cdims": cd,
            "dense_diagonal": dense_diag}


def expand(out: dict) -> np.ndarray:
    """The dense matrix a TLR output represents."""
    rd, cd = out["rdims"], out["cdims"]
    M = np.zeros((sum(rd), sum(cd)))
    r0 = 0
    for i, di in enumerate(rd):
        c0 = 0
        for j, dj in enumerate(cd):
            kind, *f = out["tiles"][(i, j)]
            M[r0:r0 + di, c0:c0 + dj] = f[0] if kind == "dense" else f[0] @ f[1].T
            c0 += dj
        r0 += di
    return M
