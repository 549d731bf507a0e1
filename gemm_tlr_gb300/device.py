"""Device memory for operands and C, and the C-ABI descriptors that point at it.

PyTorch provides the device allocations, pinned host staging and streams; the
library's kernels do every step of the product.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np

from . import _abi

_BUFS = ("U", "V", "D", "bu_U", "bu_V", "bv_U", "bv_V", "gamma")


_DTYPES = {"f32": 0, "bf16": 1, "f16": 2}   # tlr_dtype_t


def elem_bytes(dtype: str) -> int:
    return 4 if dtype == "f32" else 2


def _as_torch(a: np.ndarray, dtype: str):
    """Device-upload copy of float32 values that are exact in ``dtype``."""
    import torch
    if dtype == "bf16":
        bits = (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    if dtype == "f16":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32).astype(np.float16))
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))


def host_descriptor(X) -> tuple:
    """Descriptor with ranks only (no device pointers): for tlr_analyze and sizing."""
    d = _abi.tlr_operand_t()
    keep = []
    d.dtype = _DTYPES[X.dtype]
    d.rows, d.cols = X.rows, X.cols
    if X.kind == "dense":
        d.kind, d.ld = _abi.TLR_KIND_DENSE, X.rows
        return d, keep
    r = np.ascontiguousarray(X.ranks, dtype=np.int32)
    keep.append(r)
    d.kind, d.b, d.diag_dense, d.ranks = _abi.TLR_KIND_TLR, X.b, int(bool(X.diag_dense)), r.ctypes.data
    return d, keep


class DeviceOperand:
    """Device copy of a generator matrix (TLR or dense) plus its descriptor.

    With ``pinned=True`` a pinned host copy is kept so that ``upload`` can
    re-send the inputs host-to-device on a stream (end-to-end timing).
    """

    def __init__(self, X, device="cuda", pinned: bool = False):
        import torch
        self.X = X
        self.host = {}
        self.dev = {}
        d, keep = host_descriptor(X)
        self._keep = keep
        names = ("data",) if X.kind == "dense" else _BUFS
        for name in names:
            a = X.data if name == "data" else getattr(X, name)
            if a is None or a.size == 0:
                continue
            h = _as_torch(a, X.dtype)
            if pinned:
                h = h.pin_memory()
            self.host[name] = h
            self.dev[name] = h.to(device, non_blocking=False)
            setattr(d, name, self.dev[name].data_ptr())
        self.desc = d
        self.nbytes = sum(t.numel() * t.element_size() for t in self.dev.values())

    def upload(self, stream=None) -> int:
        """Copy the pinned host inputs to the device buffers; returns bytes copied."""
        n = 0
        for name, h in self.host.items():
            self.dev[name].copy_(h, non_blocking=True)
            n += h.numel() * h.element_size()
        return n


class DeviceProblem:
    """A ``tlr_inputs.Problem`` resident on the device, with C and a workspace."""

    def __init__(self, p, device="cuda", pinned: bool = False, workspace_bytes: Optional[int] = None,
                 fill_c_nan: bool = True):
        import torch
        self.p = p
        self.A = DeviceOperand(p.A, device, pinned)
        self.B = DeviceOperand(p.B, device, pinned)
        self.opA = _abi.TLR_OP_T if p.opA == "T" else _abi.TLR_OP_N
        self.opB = _abi.TLR_OP_T if p.opB == "T" else _abi.TLR_OP_N
        self.ldc = p.m
        if p.C is not None:
            self.C0_host = torch.from_numpy(np.ascontiguousarray(p.C, dtype=np.float32))
            if pinned:
                self.C0_host = self.C0_host.pin_memory()
            self.C0 = self.C0_host.to(device)
        else:
            self.C0_host = None
            self.C0 = None
        self.C = torch.empty(p.m * p.n, dtype=torch.float32, device=device)
        self.reset_c(fill_c_nan)
        self.handle = None
        self.plan = None
        self.ws = None
        self.ws_bytes = workspace_bytes

    def reset_c(self, fill_nan: bool = True):
        if self.C0 is not None:
            self.C.copy_(self.C0)
        else:
            self.C.fill_(float("nan") if fill_nan else 0.0)

    def make_plan(self, handle: int, budget: Optional[int] = None, order: int = _abi.TLR_ORDER_AUTO):
        import torch
        need_full = _abi.tlr_gemm_workspace_bytes_for_order(handle, self.opA, self.opB, self.A.desc, self.B.desc, 1,
                                                            order)
        if budget is None:
            budget = self.p.budget if self.p.budget is not None else need_full
        self.ws_bytes = int(budget)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=self.C.device)
        self.handle = handle
        self.plan = _abi.tlr_plan_create(handle, self.opA, self.opB, self.A.desc, self.B.desc,
                                         self.ws.data_ptr(), self.ws_bytes, order)
        return self.plan

    def run(self):
        _abi.tlr_plan_execute(self.plan, self.p.alpha, self.p.beta, self.C.data_ptr(), self.ldc)

    def info(self) -> dict:
        return _abi.tlr_plan_info(self.plan)

    def result(self) -> np.ndarray:
        """C as a (m, n) float64 numpy array."""
        return self.C.double().cpu().numpy().reshape(self.p.n, self.p.m).T

    def close(self):
        if self.plan:
            _abi.tlr_plan_destroy(self.plan)
            self.plan = None


def fake_descriptor(X, base: int) -> tuple:
    """Descriptor whose buffers sit at stand-in addresses (for host-only checks)."""
    d, keep = host_descriptor(X)
    addr = base
    names = ("data",) if X.kind == "dense" else _BUFS
    for name in names:
        a = X.data if name == "data" else getattr(X, name)
        if a is None or a.size == 0:
            continue
        setattr(d, name, addr)
        es = elem_bytes(X.dtype)
        addr += ((a.size * es + 4095) // 4096) * 4096
    return d, keep


class DeviceCompression:
    """Recompression of a dense device matrix's tiles into TLR form
    (``tlr_compress``), its outputs in device memory and, for square matrices
    with a dense diagonal, their packing into TLR buffers (``tlr_pack``).

    ``C`` is a flat float32 device tensor (m x n, column-major, leading
    dimension ``ldc``), ``omega`` a (b, s) float32 numpy array (the sketch).
    """

    def __init__(self, m: int, n: int, b: int, dense_diagonal: bool, eps: float, r_max: int, omega: np.ndarray,
                 device="cuda", batch_tiles: Optional[int] = None):
        import torch
        self.m, self.n, self.b = m, n, b
        self.nI, self.nJ = -(-m // b), -(-n // b)
        self.dense_diagonal = bool(dense_diagonal)
        self.eps, self.r_max = float(eps), int(r_max)
        self.s = int(omega.shape[1])
        assert omega.shape[0] == b
        self.omega = torch.from_numpy(np.asfortranarray(omega, dtype=np.float32).reshape(-1, order="F")).to(device)
        nt = self.nI * self.nJ
        self.U = torch.zeros(max(1, nt * b * r_max), dtype=torch.float32, device=device)
        self.V = torch.zeros_like(self.U)
        self.D = torch.zeros(max(1, self.nI * b * b if self.dense_diagonal else 1), dtype=torch.float32, device=device)
        self.ranks = torch.zeros(nt, dtype=torch.int32, device=device)
        self.errors = torch.zeros(nt, dtype=torch.float32, device=device)
        tiles = nt if batch_tiles is None else max(1, min(nt, batch_tiles))
        self.ws_bytes = _abi.tlr_compress_workspace_bytes(b, self.s, tiles)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)

    def run(self, handle: int, C, ldc: int):
        _abi.tlr_compress(handle, C.data_ptr(), ldc, self.m, self.n, self.b, self.dense_diagonal, self.eps,
                          self.r_max, self.omega.data_ptr(), self.s, self.U.data_ptr(), self.V.data_ptr(),
                          self.D.data_ptr(), self.ranks.data_ptr(), self.errors.data_ptr(), self.ws.data_ptr(),
                          self.ws_bytes)

    def dims(self):
        rd = [min(self.b, self.m - i * self.b) for i in range(self.nI)]
        cd = [min(self.b, self.n - j * self.b) for j in range(self.nJ)]
        return rd, cd

    def tiles(self) -> dict:
        """Host copy: ranks (nI, nJ), errors, and per tile ("lr", U, V) or ("dense", D) in float64."""
        b, r_max = self.b, self.r_max
        ranks = self.ranks.cpu().numpy().reshape(self.nI, self.nJ)
        errors = self.errors.cpu().numpy().astype(np.float64).reshape(self.nI, self.nJ)
        U = self.U.double().cpu().numpy()
        V = self.V.double().cpu().numpy()
        D = self.D.double().cpu().numpy()
        rd, cd = self.dims()
        tiles = {}
        for i in range(self.nI):
            for j in range(self.nJ):
                t = i * self.nJ + j
                if self.dense_diagonal and i == j:
                    tiles[(i, j)] = ("dense", D[i * b * b:(i + 1) * b * b].reshape(b, b, order="F")[:rd[i], :rd[i]])
                    continue
                r = int(ranks[i, j])
                u = U[t * b * r_max:(t + 1) * b * r_max].reshape(b, r_max, order="F")[:rd[i], :r]
                v = V[t * b * r_max:(t + 1) * b * r_max].reshape(b, r_max, order="F")[:cd[j], :r]
                tiles[(i, j)] = ("lr", u, v)
        return {"ranks": ranks, "errors": errors, "tiles": tiles, "rdims": rd, "cdims": cd,
                "dense_diagonal": self.dense_diagonal}

    def pack(self, handle: int, device="cuda"):
        """Packed fp32 TLR buffers of the result and a tlr_operand_t pointing at them:
        (descriptor, keep-alive list)."""
        import torch
        assert self.dense_diagonal and self.m == self.n
        n, b = self.n, self.b
        nt, mf, rem = self.nI, n // b, n % b
        ranks = np.ascontiguousarray(self.ranks.cpu().numpy().reshape(nt, nt), dtype=np.int32)
        R = ranks.astype(np.int64)
        inner = R[:mf, :mf].copy()
        np.fill_diagonal(inner, 0)
        size = {"U": b * inner.sum(), "V": b * inner.sum(), "D": mf * b * b}
        if rem:
            size.update({"bu_U": b * R[:mf, mf].sum(), "bu_V": rem * R[:mf, mf].sum(),
                         "bv_U": rem * R[mf, :mf].sum(), "bv_V": b * R[mf, :mf].sum(), "gamma": rem * rem})
        bufs = {k: torch.empty(max(1, int(v)), dtype=torch.float32, device=device) for k, v in size.items()}
        ptr = {k: (t.data_ptr() if size[k] > 0 else 0) for k, t in bufs.items()}
        _abi.tlr_pack(handle, n, b, self.r_max, ranks, self.U.data_ptr(), self.V.data_ptr(), self.D.data_ptr(),
                      ptr.get("U", 0), ptr.get("V", 0), ptr.get("D", 0), ptr.get("bu_U", 0), ptr.get("bu_V", 0),
                      ptr.get("bv_U", 0), ptr.get("bv_V", 0), ptr.get("gamma", 0))
        d = _abi.tlr_operand_t()
        d.kind, d.dtype, d.rows, d.cols, d.b, d.diag_dense = _abi.TLR_KIND_TLR, _DTYPES["f32"], n, n, b, 1
        r32 = np.ascontiguousarray(ranks, dtype=np.int32)
        d.ranks = r32.ctypes.data
        for k, v in ptr.items():
            if v:
                setattr(d, k, v)
        return d, [r32, bufs]
