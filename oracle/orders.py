"""Two fp64 evaluation orders of the TLR product (test infrastructure).

Used only to check the oracle's invariant that the order of evaluation does not
change the product. Both read the packed inputs through this file's own offset
code (independent of ``tlr_oracle.c`` and of the generator's packer).

* ``kblas_order``: the per-contraction-tile loop of "Tile-Low-Rank GEMM:
  Designing Storage Around the Contraction", section "Many small GEMMs": for
  each contraction tile k, coupling S = V_ik^T W_kj, right product T = S Z_kj^T,
  then the dense update C_ij += U_ik T, over all output tiles; C is updated once
  per k. The dense-tile terms are added in the same loop following the split
  A = D_A + O_A, B = D_B + O_B of "TLR Matrix Multiplication", section
  "Regular TLR GEMM".
* ``fused_k_order``: the three stages of the first page, section "One product,
  three stages", right-associative order U (S Z^T): Stage 1 one product per k
  over the stacked inner panel V_{:,k} and outer panel W_{k,:}; Stage 2 writes
  each S_ikj Z_kj^T into row block k, column block j of a terminal matrix T_i;
  Stage 3 one product per tile row, C[i,:] = alpha U_i T_i + beta C[i,:], so the
  sum over k runs inside one reduction. The dense-diagonal terms go where the
  second page puts them: O_A D_B as the k=j block V_ij^T D_jj of T_i (first half
  of "The easy terms"), D_A O_B as (D_ii W_ij) Z_ij^T, D_A D_B as D_ii D_ii.
"""
from __future__ import annotations

import numpy as np


def _dims(n, b):
    m, r = divmod(n, b)
    return [b] * m + ([r] if r else [])


class TileView:
    """Tiles of op(X) for a generator TLR or dense matrix, in fp64."""

    def __init__(self, X, op: str = "N"):
        self.X, self.op = X, op
        self.dense = X.kind == "dense"
        if self.dense:
            self.M = np.asarray(X.data, dtype=np.float64).reshape(X.rows, X.cols, order="F")
            if op == "T":
                self.M = self.M.T
            return
        b = X.b
        rd, cd = _dims(X.rows, b), _dims(X.cols, b)
        self.srd, self.scd = rd, cd
        ntr, ntc = len(rd), len(cd)
        boundary = (X.rows % b) != 0
        m = X.rows // b if boundary else None
        nr = m if boundary else ntr
        nc = m if boundary else ntc
        R = np.asarray(X.ranks, dtype=np.int64)
        self.loc = {}
        lr = lambda i, k: not (X.diag_dense and i == k)
        c = 0
        for i in range(nr):
            for k in range(nc):
                if lr(i, k):
                    self.loc[(i, k)] = ["int", c, None]
                    c += R[i, k]
        c = 0
        for k in range(nc):
            for i in range(nr):
                if lr(i, k):
                    self.loc[(i, k)][2] = c
                    c += R[i, k]
        if boundary:
            c = 0
            for i in range(m):
                self.loc[(i, m)] = ["bu", c, c]
                c += R[i, m]
            c = 0
            for j in range(m):
                self.loc[(m, j)] = ["bv", c, c]
                c += R[m, j]
        self.R, self.m, self.boundary = R, m, boundary
        self.rd, self.cd = (cd, rd) if op == "T" else (rd, cd)

    def ntr(self):
        return len(self.rd)

    def ntc(self):
        return len(self.cd)

    def _stored(self, i, k):
        X, R = self.X, self.R
        di, dk = self.srd[i], self.scd[k]
        if X.diag_dense and i == k:
            if self.boundary and i == self.m:
                D = np.asarray(X.gamma, np.float64).reshape(di, di, order="F")
            else:
                D = np.asarray(X.D[i * X.b * X.b:(i + 1) * X.b * X.b], np.float64).reshape(di, di, order="F")
            return ("dense", D)
        r = int(R[i, k])
        where, uc, vc = self.loc[(i, k)]
        if where == "int":
            Ub, Vb = X.U, X.V
        elif where == "bu":
            Ub, Vb = X.bu_U, X.bu_V
        else:
            Ub, Vb = X.bv_U, X.bv_V
        U = np.asarray(Ub[di * uc: di * (uc + r)], np.float64).reshape(di, r, order="F")
        V = np.asarray(Vb[dk * vc: dk * (vc + r)], np.float64).reshape(dk, r, order="F")
        return ("lr", U, V)

    def tile(self, i, k):
        """('lr', U, V) with op(X)_ik = U V^T, or ('dense', D)."""
        if self.dense:
            raise RuntimeError("dense operands are read as whole row blocks")
        if self.op == "N":
            return self._stored(i, k)
        t = self._stored(k, i)
        if t[0] == "dense":
            return ("dense", t[1].T)
        return ("lr", t[2], t[1])


def kblas_order(A, B, opA, opB, alpha, beta, C, ldc):
    """Per-contraction-tile loop; returns C_out (fp64, rows x cols)."""
    Av, Bv = TileView(A, opA), TileView(B, opB)
    if Av.dense:
        raise ValueError("left operand must be TLR")
    rd = Av.rd
    kd = Av.cd
    if Bv.dense:
        ncols = Bv.M.shape[1]
        cd = [ncols]
    else:
        cd = Bv.cd
    M, N = sum(rd), sum(cd)
    out = np.zeros((M, N))
    if beta != 0.0:
        out[:] = beta * np.asarray(C, np.float64).reshape(-1)[: ldc * N].reshape(N, ldc).T[:M, :]
    ro = np.cumsum([0] + rd)
    co = np.cumsum([0] + list(cd))
    ko = np.cumsum([0] + kd)
    for k in range(len(kd)):
        for i in range(len(rd)):
            a = Av.tile(i, k)
            for j in range(len(cd)):
                if Bv.dense:
                    Bkj = Bv.M[ko[k]:ko[k + 1], :]
                    if a[0] == "dense":
                        upd = a[1] @ Bkj
                    else:
                        upd = a[1] @ (a[2].T @ Bkj)
                else:
                    bt = Bv.tile(k, j)
                    if a[0] == "lr" and bt[0] == "lr":
                        S = a[2].T @ bt[1]            # coupling
                        T = S @ bt[2].T               # right product
                        upd = a[1] @ T                # dense update
                    elif a[0] == "dense" and bt[0] == "lr":
                        upd = (a[1] @ bt[1]) @ bt[2].T
                    elif a[0] == "lr" and bt[0] == "dense":
                        upd = a[1] @ (a[2].T @ bt[1])
                    else:
                        upd = a[1] @ bt[1]
                out[ro[i]:ro[i + 1], co[j]:co[j + 1]] += alpha * upd
    return out


def fused_k_order(A, B, opA, opB, alpha, beta, C, ldc):
    """Three-stage right-associative order with k inside one reduction; fp64."""
    Av, Bv = TileView(A, opA), TileView(B, opB)
    if Av.dense:
        raise ValueError("left operand must be TLR")
    rd, kd = Av.rd, Av.cd
    nI, nK = len(rd), len(kd)
    ko = np.cumsum([0] + kd)
    if Bv.dense:
        N = Bv.M.shape[1]
        cd = [N]
    else:
        cd = Bv.cd
        N = sum(cd)
    nJ = len(cd)
    co = np.cumsum([0] + list(cd))
    M = sum(rd)
    ro = np.cumsum([0] + rd)
    out = np.zeros((M, N))
    Cf = None
    if beta != 0.0:
        Cf = np.asarray(C, np.float64).reshape(-1)[: ldc * N].reshape(N, ldc).T[:M, :]
    A_lr = {(i, k): Av.tile(i, k) for i in range(nI) for k in range(nK)}
    # Stage 1: for each k one product over the stacked panels (dense B: the row block B_k)
    S = {}
    for k in range(nK):
        rows = [i for i in range(nI) if A_lr[(i, k)][0] == "lr"]
        if not rows:
            continue
        Vk = np.hstack([A_lr[(i, k)][2] for i in rows])            # d_k x sigma_k
        if Bv.dense:
            S[k] = (rows, None, Vk.T @ Bv.M[ko[k]:ko[k + 1], :])
            continue
        cols = [j for j in range(nJ) if Bv.tile(k, j)[0] == "lr"]
        if not cols:
            continue
        Wk = np.hstack([Bv.tile(k, j)[1] for j in cols])           # d_k x Gamma_k
        S[k] = (rows, cols, Vk.T @ Wk)
    # Stage 2: terminal matrices T_i (row block k has height r_ik)
    Ti = {}
    for i in range(nI):
        ks = [k for k in range(nK) if A_lr[(i, k)][0] == "lr"]
        rk = [A_lr[(i, k)][1].shape[1] for k in ks]
        T = np.zeros((sum(rk), N))
        off = 0
        for k, r in zip(ks, rk):
            if Bv.dense:
                rows, _, Sk = S[k]
                a0 = sum(A_lr[(ii, k)][1].shape[1] for ii in rows[:rows.index(i)])
                T[off:off + r, :] = Sk[a0:a0 + r, :]
            else:
                for j in range(nJ):
                    bt = Bv.tile(k, j)
                    if bt[0] == "lr":
                        rows, cols, Sk = S[k]
                        a0 = sum(A_lr[(ii, k)][1].shape[1] for ii in rows[:rows.index(i)])
                        b0 = sum(Bv.tile(k, jj)[1].shape[1] for jj in cols[:cols.index(j)])
                        Sikj = Sk[a0:a0 + r, b0:b0 + bt[1].shape[1]]
                        T[off:off + r, co[j]:co[j + 1]] = Sikj @ bt[2].T
                    else:  # k == j, dense B tile: V_ij^T D_jj
                        T[off:off + r, co[j]:co[j + 1]] = A_lr[(i, k)][2].T @ bt[1]
            off += r
        Ti[i] = (ks, T)
    # Stage 3: one product per tile row over the packed outer panel, plus D_A terms
    for i in range(nI):
        ks, T = Ti[i]
        acc = np.zeros((rd[i], N))
        if ks:
            Ui = np.hstack([A_lr[(i, k)][1] for k in ks])          # d_i x rho_i
            acc += Ui @ T
        for k in range(nK):
            if A_lr[(i, k)][0] != "dense":
                continue
            Dii = A_lr[(i, k)][1]
            if Bv.dense:
                acc += Dii @ Bv.M[ko[k]:ko[k + 1], :]
                continue
            for j in range(nJ):
                bt = Bv.tile(k, j)
                if bt[0] == "lr":
                    acc[:, co[j]:co[j + 1]] += (Dii @ bt[1]) @ bt[2].T
                else:
                    acc[:, co[j]:co[j + 1]] += Dii @ bt[1]
        out[ro[i]:ro[i + 1], :] = alpha * acc + (beta * Cf[ro[i]:ro[i + 1], :] if Cf is not None else 0.0)
    return out
