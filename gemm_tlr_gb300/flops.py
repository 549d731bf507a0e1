"""Executed FLOP count of a planned product, from ranks alone.

"Executed FLOPs" are the products the method runs, 2*M*N*K each at logical
ranks ("Tile-Low-Rank GEMM: Designing Storage Around the Contraction", section
"Results": throughput is reported on executed FLOPs). For the right-associative
order U (S Z^T) with op(A) = X, op(B) = Y:

  Stage 1   sum_k 2 sigma_k Gamma_k d_k              S_k = V_{:,k}^T W_{k,:}
  Stage 2   sum_{k,j} 2 sigma_k d_j r^Y_kj            T_i blocks S_ikj Z_kj^T
  Stage 3   sum_i 2 d_i N rho_i                       U_i T_i, the sum over k inside K
  dense     sum_j 2 sigma_j d_j^2 (V_jj^T D_jj)  +  sum_i 2 d_i Gamma_i d_i (D_ii W_i,:)
            + sum_{i, j != i} 2 d_i d_j r^Y_ij (P_ij Z_ij^T) + sum_i 2 d_i^3 (D_ii D_ii)

(the dense-tile terms follow "TLR Matrix Multiplication", section "Regular TLR
GEMM"). With a dense Y, Stage 1 is sum_k 2 sigma_k N d_k, there is no Stage 2,
and the dense term is sum_i 2 d_i N d_i. The split into rectangles does not
change the count (each term is bilinear in the row and column sets).
"""
from __future__ import annotations

import numpy as np


def _dims(n, b):
    m, r = divmod(n, b)
    return [b] * m + ([r] if r else [])


def _logical(X, op):
    """(ranks, dense-tile mask, row dims, col dims) of op(X) for a TLR matrix."""
    R = np.asarray(X.ranks, dtype=np.int64)
    rd, cd = _dims(X.rows, X.b), _dims(X.cols, X.b)
    dense = np.zeros(R.shape, dtype=bool)
    if X.diag_dense:
        for t in range(min(R.shape)):
            dense[t, t] = True
    R = np.where(dense, 0, R)
    if op == "T":
        return R.T, dense.T, cd, rd
    return R, dense, rd, cd


def executed_flops(p, order: str = "R") -> dict:
    """Executed FLOPs of the right ("R") or left ("L") order for the whole of C.

    The left order (U S) Z^T is the right order of the transposed product
    C^T = op(B)^T op(A)^T, which is how the library evaluates it.
    """
    if order == "R":
        return executed_flops_right(p)
    if p.A.kind == "dense" or p.B.kind == "dense":
        raise ValueError("with a dense operand only one order exists")
    flip = {"N": "T", "T": "N"}
    q = _Swapped(p.B, flip[p.opB], p.A, flip[p.opA], p.n)
    return executed_flops_right(q)


class _Swapped:
    def __init__(self, A, opA, B, opB, n):
        self.A, self.opA, self.B, self.opB, self.n = A, opA, B, opB, n


def executed_flops_right(p) -> dict:
    X = _logical(p.A, p.opA)
    RX, DX, rdX, cdX = X
    sig = RX.sum(axis=0)
    rho = RX.sum(axis=1)
    out = {"stage1": 0.0, "stage2": 0.0, "stage3": 0.0, "dense": 0.0}
    if p.B.kind == "dense":
        N = p.n
        out["stage1"] = float(sum(2.0 * sig[k] * N * cdX[k] for k in range(len(cdX))))
        out["stage3"] = float(sum(2.0 * rdX[i] * N * rho[i] for i in range(len(rdX))))
        out["dense"] = float(sum(2.0 * rdX[i] * N * cdX[i] for i in range(len(rdX)) if DX[i, i]))
    else:
        RY, DY, rdY, cdY = _logical(p.B, p.opB)
        Gam = RY.sum(axis=1)
        N = sum(cdY)
        out["stage1"] = float(sum(2.0 * sig[k] * Gam[k] * cdX[k] for k in range(len(cdX))))
        out["stage2"] = float(sum(2.0 * sig[k] * cdY[j] * RY[k, j]
                                  for k in range(RY.shape[0]) for j in range(RY.shape[1]) if not DY[k, j]))
        out["stage3"] = float(sum(2.0 * rdX[i] * N * rho[i] for i in range(len(rdX))))
        d = 0.0
        for j in range(len(cdY)):
            if j < RY.shape[0] and DY[j, j]:
                d += 2.0 * sig[j] * cdY[j] * rdY[j]
        for i in range(len(rdX)):
            if i < RX.shape[1] and DX[i, i]:
                d += 2.0 * rdX[i] * Gam[i] * cdX[i]
                for j in range(len(cdY)):
                    if DY[i, j]:
                        d += 2.0 * rdX[i] * cdY[j] * cdX[i]
                    else:
                        d += 2.0 * rdX[i] * cdY[j] * RY[i, j]
        out["dense"] = d
    out["total"] = out["stage1"] + out["stage2"] + out["stage3"] + out["dense"]
    return out
