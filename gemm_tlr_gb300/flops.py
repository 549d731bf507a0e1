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
and the dense term is sum_i 2 d_i N d_i. For one order the split into
rectangles does not change the count (each term is bilinear in the row and
column sets); a plan that takes the cheaper order per rectangle is counted
rectangle by rectangle (`executed_flops_rects`), each term restricted to the
rectangle's tile rows I and tile columns J (sigma_k and Gamma_k become the rank
sums over I and J, N becomes W_J).
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
    """Executed FLOPs of the right ("R"), left ("L") or per-triple ("P") order for the whole of C.

    The left order (U S) Z^T is the right order of the transposed product
    C^T = op(B)^T op(A)^T, which is how the library evaluates it.
    """
    return executed_flops_rect(p, order)


def _grid(p):
    """Tile counts of C's rows and columns."""
    b = p.A.b if p.A.kind == "tlr" else p.B.b
    return len(_dims(p.m, b)), len(_dims(p.n, b))


def executed_flops_rect(p, order: str, I=None, J=None) -> dict:
    """Executed FLOPs of one rectangle of C (tile rows I, tile columns J; all by
    default) under order "R", "L" or "P" (per tile triple)."""
    nI, nJ = _grid(p)
    I = range(nI) if I is None else I
    J = range(nJ) if J is None else J
    if order == "R":
        if p.A.kind == "dense":
            raise ValueError("a dense left operand has only the left order")
        return executed_flops_right(p, I, J)
    if order == "P":
        return executed_flops_triple(p, I, J)
    if order != "L":
        raise ValueError(order)
    if p.B.kind == "dense":
        raise ValueError("a dense right operand has only the right order")
    flip = {"N": "T", "T": "N"}
    q = _Swapped(p.B, flip[p.opB], p.A, flip[p.opA], p.n)
    return executed_flops_right(q, J, I)


def executed_flops_triple(p, I=None, J=None) -> dict:
    """The per-triple order ("TLR Matrix Multiplication", section "The O_A O_B
    terms"): after S_ikj = V_ik^T W_kj, a triple with r_ik <= r_kj forms
    S_ikj Z_kj^T and adds U_ik times it (K = r_ik), otherwise it forms U_ik S_ikj
    and adds it times Z_kj^T (K = r_kj). Stage 1 and the dense-tile terms are
    those of the right order; the k = j block V_ij^T D_jj joins the final
    product with K = r_ij. Counted from the rule alone (a plan may move a few
    triples to the other side so that a tile's K-loop stays within its segment
    limit; it never does for rank maps that decay with |i - j|)."""
    if p.A.kind != "tlr" or p.B.kind != "tlr":
        raise ValueError("the per-triple order needs two TLR operands")
    RX, DX, rdX, cdX = _logical(p.A, p.opA)
    RY, DY, rdY, cdY = _logical(p.B, p.opB)
    I = list(range(len(rdX))) if I is None else list(I)
    J = list(range(len(cdY))) if J is None else list(J)
    base = executed_flops_right(p, I, J)
    out = {"stage1": base["stage1"], "dense": base["dense"], "stage2": 0.0, "stage3": 0.0}
    nk = RX.shape[1]
    for i in I:
        for j in J:
            for k in range(nk):
                if DX[i, k]:
                    continue                      # k = i: P_ij Z_ij^T, a dense-tile term
                if DY[k, j]:
                    out["stage3"] += 2.0 * rdX[i] * cdY[j] * RX[i, k]        # U_ij (V_ij^T D_jj)
                    continue
                ra, rb = int(RX[i, k]), int(RY[k, j])
                if ra == 0 or rb == 0:
                    continue
                if ra <= rb:
                    out["stage2"] += 2.0 * ra * cdY[j] * rb                  # S_ikj Z_kj^T
                    out["stage3"] += 2.0 * rdX[i] * cdY[j] * ra
                else:
                    out["stage2"] += 2.0 * rdX[i] * ra * rb                  # U_ik S_ikj
                    out["stage3"] += 2.0 * rdX[i] * cdY[j] * rb
    out["total"] = out["stage1"] + out["stage2"] + out["stage3"] + out["dense"]
    return out


def executed_flops_rects(p, rects) -> dict:
    """Sum over a plan's rectangles [(i0, i1, j0, j1, order)], each with its own order."""
    tot = {"stage1": 0.0, "stage2": 0.0, "stage3": 0.0, "dense": 0.0, "total": 0.0}
    for (i0, i1, j0, j1, order) in rects:
        f = executed_flops_rect(p, order, range(i0, i1), range(j0, j1))
        for k in tot:
            tot[k] += f[k]
    return tot


class _Swapped:
    def __init__(self, A, opA, B, opB, n):
        self.A, self.opA, self.B, self.opB, self.n = A, opA, B, opB, n


def executed_flops_right(p, I=None, J=None) -> dict:
    """Right order U (S Z^T) on tile rows I x tile columns J of C (all of C by default)."""
    X = _logical(p.A, p.opA)
    RX, DX, rdX, cdX = X
    I = list(range(len(rdX))) if I is None else list(I)
    sig = RX[I, :].sum(axis=0)                 # sigma_k over the rectangle's tile rows
    rho = RX.sum(axis=1)
    out = {"stage1": 0.0, "stage2": 0.0, "stage3": 0.0, "dense": 0.0}
    if p.B.kind == "dense":
        cdY = _dims(p.n, p.A.b)                # the dense operand's columns in tiles of the TLR one
        J = list(range(len(cdY))) if J is None else list(J)
        W = sum(cdY[j] for j in J)
        out["stage1"] = float(sum(2.0 * sig[k] * W * cdX[k] for k in range(len(cdX))))
        out["stage3"] = float(sum(2.0 * rdX[i] * W * rho[i] for i in I))
        out["dense"] = float(sum(2.0 * rdX[i] * W * cdX[i] for i in I if DX[i, i]))
    else:
        RY, DY, rdY, cdY = _logical(p.B, p.opB)
        J = list(range(len(cdY))) if J is None else list(J)
        Gam = RY[:, J].sum(axis=1)             # Gamma_k over the rectangle's tile columns
        W = sum(cdY[j] for j in J)
        out["stage1"] = float(sum(2.0 * sig[k] * Gam[k] * cdX[k] for k in range(len(cdX))))
        out["stage2"] = float(sum(2.0 * sig[k] * cdY[j] * RY[k, j]
                                  for k in range(RY.shape[0]) for j in J if not DY[k, j]))
        out["stage3"] = float(sum(2.0 * rdX[i] * W * rho[i] for i in I))
        d = 0.0
        for j in J:
            if j < RY.shape[0] and DY[j, j]:
                d += 2.0 * sig[j] * cdY[j] * rdY[j]
        for i in I:
            if i < RX.shape[1] and DX[i, i]:
                d += 2.0 * rdX[i] * Gam[i] * cdX[i]
                for j in J:
                    if DY[i, j]:
                        d += 2.0 * rdX[i] * cdY[j] * cdX[i]
                    else:
                        d += 2.0 * rdX[i] * cdY[j] * RY[i, j]
        out["dense"] = d
    out["total"] = out["stage1"] + out["stage2"] + out["stage3"] + out["dense"]
    return out
