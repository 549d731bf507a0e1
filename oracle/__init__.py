"""CPU fp64 oracle for the Tile-Low-Rank GEMM (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the GPU path
(``gemm_tlr_gb300``) and never imports it; both sides take their inputs from the
seeded generator module ``tlr_inputs``, which holds none of the method's
arithmetic.

Contents
--------
* ``tlr_oracle.c`` (loaded here through ctypes): the plain definition
  ``C <- alpha op(A) op(B) + beta C`` with every TLR operand expanded tile by tile
  and every output entry summed in fp64 over the contraction index in ascending
  order ("Tile-Low-Rank GEMM: Designing Storage Around the Contraction", opening
  section and section "Many small GEMMs"; "TLR Matrix Multiplication", section
  "Introduction: TLR GEMM").
* ``orders.py``: two evaluation orders of the same product in fp64 -- the
  per-contraction-tile loop with three batched products per step (first page,
  section "Many small GEMMs") and the fused-k three-stage order (first page,
  section "One product, three stages"), plus the dense/low-rank split of the
  second page (section "Regular TLR GEMM"). They exist to check the invariant
  that both orders give the definition's result.
* ``planner_ref.py``: the rank-metadata quantities the planner is built on,
  written from their definitions (first page, section "Association order and
  workspace").
* ``tlr_output.py``: the TLR-output product -- the dense product tiles
  recompressed tile by tile to the smallest rank within a relative Frobenius
  tolerance (second page, section "Introduction: TLR GEMM"; the recompression
  rule is a reading, stated there). It has no GPU counterpart yet.

Every function here is pinned by a ``-m "not gpu"`` test against something other
than itself (brute force on tiny inputs, closed forms, special cases, printed
values of the worked example); see ``tests/test_oracle.py`` and
``tests/test_tlr_output_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tlr_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libtlr_oracle.so")
_lib = None
_lock = threading.Lock()


def _compile(out: str, defines=()) -> None:
    cc = os.environ.get("CC", "gcc")
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call([cc, "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           *[f"-D{d}" for d in defines], _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, out)


def build(force: bool = False) -> str:
    """Compile the C oracle (plain C, OpenMP) next to its source."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        _compile(_LIB_PATH)
    return _LIB_PATH


def load_mutant(code: int, directory: str):
    """Load a copy of the oracle with a planted mistake (pin tests only)."""
    global _lib
    path = os.path.join(directory, f"libtlr_oracle_mut{code}.so")
    _compile(path, [f"ORC_MUTATE={code}"])
    return path


class use_library:
    """Context manager: route this module's calls through another build of the oracle."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = _lib
        _lib = None
        _load(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


class _Mat(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32), ("diag_dense", ctypes.c_int32),
        ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("b", ctypes.c_int64),
        ("ranks", ctypes.c_void_p),
        ("U", ctypes.c_void_p), ("V", ctypes.c_void_p), ("D", ctypes.c_void_p),
        ("bu_U", ctypes.c_void_p), ("bu_V", ctypes.c_void_p),
        ("bv_U", ctypes.c_void_p), ("bv_V", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
        ("dense", ctypes.c_void_p), ("ld", ctypes.c_int64),
    ]


def _load(path: Optional[str] = None):
    global _lib
    with _lock:
        if _lib is None:
            if path is None:
                path = build()
            lib = ctypes.CDLL(path)
            lib.orc_gemm_block.restype = ctypes.c_int
            lib.orc_gemm_block.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.POINTER(_Mat),
                ctypes.POINTER(_Mat), ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            lib.orc_expand_tile.restype = ctypes.c_int
            lib.orc_expand_tile.argtypes = [ctypes.POINTER(_Mat), ctypes.c_int, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64]
            lib.orc_check.restype = ctypes.c_int
            lib.orc_check.argtypes = [ctypes.POINTER(_Mat)]
            lib.orc_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(a) -> Optional[np.ndarray]:
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a) -> Optional[int]:
    return None if a is None else a.ctypes.data


def _mat(X):
    """ctypes descriptor for a generator matrix; returns (struct, keep-alive list)."""
    keep = []
    m = _Mat()
    if X.kind == "dense":
        d = _f32(X.data)
        keep.append(d)
        m.kind, m.rows, m.cols, m.dense, m.ld = 1, X.rows, X.cols, _ptr(d), X.rows
        return m, keep
    ranks = np.ascontiguousarray(X.ranks, dtype=np.int32)
    keep.append(ranks)
    m.kind, m.diag_dense = 0, int(bool(X.diag_dense))
    m.rows, m.cols, m.b = X.rows, X.cols, X.b
    m.ranks = ranks.ctypes.data
    for name in ("U", "V", "D", "bu_U", "bu_V", "bv_U", "bv_V", "gamma"):
        a = _f32(getattr(X, name))
        keep.append(a)
        setattr(m, name, _ptr(a))
    return m, keep


def num_threads() -> int:
    return int(_load().orc_num_threads())


def check(X) -> int:
    m, keep = _mat(X)
    return int(_load().orc_check(ctypes.byref(m)))


def expand_tile(X, ti: int, tk: int, op: str = "N") -> np.ndarray:
    """Dense tile (ti, tk) of op(X) in fp64."""
    lib = _load()
    m, keep = _mat(X)
    rd = [X.b] * (X.rows // X.b) + ([X.rows % X.b] if X.rows % X.b else [])
    cd = [X.b] * (X.cols // X.b) + ([X.cols % X.b] if X.cols % X.b else [])
    if op == "T":
        rd, cd = cd, rd
    out = np.zeros((rd[ti], cd[tk]), dtype=np.float64, order="F")
    rc = lib.orc_expand_tile(ctypes.byref(m), 1 if op == "T" else 0, ti, tk, out.ctypes.data, rd[ti])
    if rc:
        raise ValueError(f"orc_expand_tile failed: {rc}")
    return out


def gemm_block(A, B, opA: str, opB: str, alpha: float, beta: float, C: Optional[np.ndarray],
               ldc: int, rows: Sequence[int], cols: Sequence[int]) -> np.ndarray:
    """Entries C_out[rows, cols] (fp64, shape len(rows) x len(cols)).

    ``C`` is the full input C (column-major, leading dimension ``ldc``) or None
    when beta == 0 (it is then never read).
    """
    lib = _load()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    nr, nc = rows.size, cols.size
    ma, ka = _mat(A)
    mb, kb = _mat(B)
    cin = None
    if beta != 0.0:
        if C is None:
            raise ValueError("beta != 0 needs C")
        flat = np.asarray(C, dtype=np.float32).reshape(-1)
        sub = flat[rows[:, None] + cols[None, :] * ldc]          # (nr, nc)
        cin = np.ascontiguousarray(sub.T).reshape(-1)            # column-major block
    out = np.empty(nr * nc, dtype=np.float64)
    rc = lib.orc_gemm_block(1 if opA == "T" else 0, 1 if opB == "T" else 0, float(alpha),
                            ctypes.byref(ma), ctypes.byref(mb), float(beta),
                            rows.ctypes.data, nr, cols.ctypes.data, nc,
                            None if cin is None else cin.ctypes.data, out.ctypes.data)
    if rc:
        raise ValueError(f"orc_gemm_block failed with code {rc}")
    return out.reshape(nc, nr).T  # (nr, nc)


def gemm_problem(p, rows: Optional[Sequence[int]] = None, cols: Optional[Sequence[int]] = None) -> np.ndarray:
    """Oracle result for a ``tlr_inputs.Problem`` (all of C, or a sampled block)."""
    rows = np.arange(p.m) if rows is None else rows
    cols = np.arange(p.n) if cols is None else cols
    return gemm_block(p.A, p.B, p.opA, p.opB, p.alpha, p.beta, p.C, p.m, rows, cols)
