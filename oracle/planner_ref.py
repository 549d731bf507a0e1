"""Rank-metadata quantities written from their definitions (test infrastructure).

"Tile-Low-Rank GEMM: Designing Storage Around the Contraction", section
"Association order and workspace": with rho_i = sum_k r^A_ik and
gamma_j = sum_k r^B_kj, the right-associative order U (S Z^T) ends with one
product per tile row of C and the left-associative order (U S) Z^T with one per
tile column. Their final-stage costs (the formula itself did not survive
extraction; this is the reading that reproduces the page's printed
F_R = 2 b^2 * 528 and F_L = 2 b^2 * 608 for the worked example) are

    F_R = sum_{i in I} 2 * d_i * W_J * rho_i,    W_J = sum_{j in J} d_j
    F_L = sum_{j in J} 2 * d_j * H_I * gamma_j,  H_I = sum_{i in I} d_i

and the terminal workspaces are (sum_i rho_i) x W_J for the right order and
H_I x (sum_j gamma_j) for the left order. Stage 1 for contraction tile k is one
product of shape (sigma_k, Gamma_k, d_k) with sigma_k = sum_i r^A_ik and
Gamma_k = sum_j r^B_kj (section "One product, three stages", Stage 1).
"""
from __future__ import annotations

import numpy as np


def lowrank_mask(ranks: np.ndarray, diag_dense: bool) -> np.ndarray:
    m = np.ones(ranks.shape, dtype=bool)
    if diag_dense:
        for t in range(min(ranks.shape)):
            m[t, t] = False
    return m


def metadata(rA: np.ndarray, rB: np.ndarray, dA_rows, dK, dB_cols, diag_dense_A=False, diag_dense_B=False):
    """Quantities of the worked example, for whole C (I = all rows, J = all columns)."""
    rA = np.asarray(rA, np.int64) * lowrank_mask(np.asarray(rA), diag_dense_A)
    rB = np.asarray(rB, np.int64) * lowrank_mask(np.asarray(rB), diag_dense_B)
    rho = rA.sum(axis=1)
    gamma = rB.sum(axis=0)
    sigma = rA.sum(axis=0)
    Gam = rB.sum(axis=1)
    W = int(sum(dB_cols))
    H = int(sum(dA_rows))
    F_R = int(sum(2 * dA_rows[i] * W * rho[i] for i in range(len(rho))))
    F_L = int(sum(2 * dB_cols[j] * H * gamma[j] for j in range(len(gamma))))
    stage1 = [(int(sigma[k]), int(Gam[k]), int(dK[k])) for k in range(len(dK))]
    products = [(int(rA[i, k]), int(rB[k, j]))
                for i in range(rA.shape[0]) for k in range(rA.shape[1]) for j in range(rB.shape[1])
                if rA[i, k] > 0 and rB[k, j] > 0]
    stage3_R = [(int(dA_rows[i]), W, int(rho[i])) for i in range(len(rho))]
    return {
        "rho": [int(x) for x in rho], "gamma": [int(x) for x in gamma],
        "sigma": [int(x) for x in sigma], "Gamma": [int(x) for x in Gam],
        "F_R": F_R, "F_L": F_L,
        "order": "R" if F_R <= F_L else "L",
        "T_R": (int(rho.sum()), W), "T_L": (H, int(gamma.sum())),
        "stage1": stage1, "coupling_products": len(products),
        "distinct_shapes": len(set(products)), "stage3_R": stage3_R,
    }
