"""ctypes binding of ``include/tlr_gemm.h`` (argument marshalling only).

Every function here forwards to the entry point of the same name in
``libtlrgemm.so``; all work runs in the library's CUDA kernels. Loading fails
loudly when the library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtlrgemm.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "tlr_gemm.h")

TLR_OP_N, TLR_OP_T = 0, 1
TLR_F32, TLR_BF16, TLR_F16 = 0, 1, 2
TLR_KIND_TLR, TLR_KIND_DENSE = 0, 1
TLR_ORDER_AUTO, TLR_ORDER_RIGHT, TLR_ORDER_LEFT, TLR_ORDER_TRIPLE, TLR_ORDER_PER_RECT = 0, 1, 2, 3, 4
STATUS = {0: "OK", 1: "INVALID_ARG", 2: "ALIGNMENT", 3: "WORKSPACE_TOO_SMALL", 4: "UNSUPPORTED",
          5: "CUDA_ERROR", 6: "TIMEOUT", 7: "NOT_INITIALIZED"}
KIND_STAGE1, KIND_STAGE2, KIND_STAGE3, KIND_ROUND, KIND_SCALE = 0, 1, 2, 3, 4


class TLRError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: TLR_STATUS_{STATUS.get(code, code)}")
        self.code = code


class tlr_operand_t(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
        ("b", ctypes.c_int32), ("diag_dense", ctypes.c_int32),
        ("ranks", ctypes.c_void_p), ("u_offsets", ctypes.c_void_p), ("v_offsets", ctypes.c_void_p),
        ("U", ctypes.c_void_p), ("V", ctypes.c_void_p), ("D", ctypes.c_void_p),
        ("bu_U", ctypes.c_void_p), ("bu_V", ctypes.c_void_p),
        ("bv_U", ctypes.c_void_p), ("bv_V", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
        ("data", ctypes.c_void_p), ("ld", ctypes.c_int64),
    ]


class tlr_plan_info_t(ctypes.Structure):
    _fields_ = [
        ("runs", ctypes.c_int32), ("runs_right", ctypes.c_int32), ("runs_left", ctypes.c_int32),
        ("runs_triple", ctypes.c_int32), ("launches", ctypes.c_int64),
        ("flops_executed", ctypes.c_double), ("flops_stage1", ctypes.c_double),
        ("flops_stage2", ctypes.c_double), ("flops_stage3", ctypes.c_double),
        ("flops_dense_terms", ctypes.c_double), ("flops_right_final", ctypes.c_double),
        ("flops_left_final", ctypes.c_double), ("workspace_bytes", ctypes.c_size_t),
        ("tasks", ctypes.c_int64), ("flops_launch", ctypes.c_double * 3),
    ]


class tlr_rect_t(ctypes.Structure):
    _fields_ = [("i0", ctypes.c_int32), ("i1", ctypes.c_int32), ("j0", ctypes.c_int32), ("j1", ctypes.c_int32),
                ("order", ctypes.c_int32)]


class tlr_analysis_t(ctypes.Structure):
    _fields_ = [
        ("nt_i", ctypes.c_int32), ("nt_k", ctypes.c_int32), ("nt_j", ctypes.c_int32),
        ("rho", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("sigma", ctypes.c_void_p),
        ("Gamma", ctypes.c_void_p), ("stage1_mnk", ctypes.c_void_p), ("stage3_mnk", ctypes.c_void_p),
        ("F_R", ctypes.c_double), ("F_L", ctypes.c_double), ("order", ctypes.c_int32),
        ("T_right_rows", ctypes.c_int64), ("T_right_cols", ctypes.c_int64),
        ("T_left_rows", ctypes.c_int64), ("T_left_cols", ctypes.c_int64),
        ("coupling_products", ctypes.c_int64), ("distinct_shapes", ctypes.c_int64),
        ("F_P", ctypes.c_double),
    ]


_P = ctypes.c_void_p
_OP = ctypes.POINTER(tlr_operand_t)
_SIGS = {
    "tlr_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tlr_create": (ctypes.c_int, [ctypes.POINTER(_P), _P]),
    "tlr_destroy": (ctypes.c_int, [_P]),
    "tlr_set_stream": (ctypes.c_int, [_P, _P]),
    "tlr_analyze": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _OP, _OP, ctypes.POINTER(tlr_analysis_t)]),
    "tlr_gemm_workspace_bytes": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, _OP, _OP, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_size_t)]),
    "tlr_gemm_workspace_bytes_for_order": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, _OP, _OP, ctypes.c_int,
                                                          ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "tlr_plan_create": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, _OP, _OP, _P, ctypes.c_size_t,
                                       ctypes.c_int, ctypes.POINTER(_P)]),
    "tlr_plan_info": (ctypes.c_int, [_P, ctypes.POINTER(tlr_plan_info_t)]),
    "tlr_plan_rects": (ctypes.c_int, [_P, ctypes.POINTER(tlr_rect_t), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "tlr_debug_plan_rects": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _OP, _OP, ctypes.c_size_t, ctypes.c_int,
                                            ctypes.POINTER(tlr_rect_t), ctypes.c_int32,
                                            ctypes.POINTER(ctypes.c_int32)]),
    "tlr_plan_execute": (ctypes.c_int, [_P, ctypes.c_float, ctypes.c_float, _P, ctypes.c_int64]),
    "tlr_plan_destroy": (ctypes.c_int, [_P]),
    "tlr_gemm": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, ctypes.c_float, _OP, _OP, ctypes.c_float,
                                _P, ctypes.c_int64, _P, ctypes.c_size_t]),
    "tlr_gemm_static_scratch": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, ctypes.c_float, _OP, _OP,
                                               ctypes.c_float, _P, ctypes.c_int64]),
    "tlr_get_device_status": (ctypes.c_int, [_P]),
    "tlr_set_timing": (ctypes.c_int, [_P, ctypes.c_int]),
    "tlr_get_timing": (ctypes.c_int, [_P, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_int64)]),
    "tlr_reset_timing": (ctypes.c_int, [_P]),
    "tlr_set_wait_limit_us": (ctypes.c_int, [_P, ctypes.c_int64]),
    "tlr_debug_check_plan": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _OP, _OP, ctypes.c_size_t, ctypes.c_int,
                                            ctypes.POINTER(tlr_plan_info_t), ctypes.c_char_p, ctypes.c_size_t]),
    "tlr_debug_unsatisfied_wait": (ctypes.c_int, [_P]),
    "tlr_compress_workspace_bytes": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int64,
                                                    ctypes.POINTER(ctypes.c_size_t)]),
    "tlr_compress": (ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_int32, ctypes.c_float, ctypes.c_int32, _P, ctypes.c_int32,
                                    _P, _P, _P, _P, _P, _P, ctypes.c_size_t]),
    "tlr_pack": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P,
                                _P, _P, _P, _P, _P]),
}

_lib = None
_lock = threading.Lock()


def header_symbols():
    """Names of the functions declared in include/tlr_gemm.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(tlr_[a-z_0-9]+)\s*\(", text)))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                    "(the library has no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def check(code: int, what: str):
    if code != 0:
        raise TLRError(code, what)


# ------------------------------------------------------------------ same-name wrappers
def tlr_status_string(code: int) -> str:
    return lib().tlr_status_string(code).decode()


def tlr_create(stream: int = 0) -> int:
    h = _P()
    check(lib().tlr_create(ctypes.byref(h), _P(stream)), "tlr_create")
    return h.value


def tlr_destroy(h: int) -> None:
    check(lib().tlr_destroy(_P(h)), "tlr_destroy")


def tlr_set_stream(h: int, stream: int) -> None:
    check(lib().tlr_set_stream(_P(h), _P(stream)), "tlr_set_stream")


def tlr_analyze(opA: int, opB: int, A: tlr_operand_t, B: tlr_operand_t, nt_i: int, nt_k: int, nt_j: int):
    import numpy as np
    arrs = {k: np.zeros(n, dtype=np.int64) for k, n in
            (("rho", nt_i), ("gamma", nt_j), ("sigma", nt_k), ("Gamma", nt_k),
             ("stage1_mnk", 3 * nt_k), ("stage3_mnk", 3 * nt_i))}
    a = tlr_analysis_t()
    for k, v in arrs.items():
        setattr(a, k, v.ctypes.data)
    check(lib().tlr_analyze(opA, opB, ctypes.byref(A), ctypes.byref(B), ctypes.byref(a)), "tlr_analyze")
    out = {k: v for k, v in arrs.items()}
    for f, _ in tlr_analysis_t._fields_:
        if f not in arrs:
            out[f] = getattr(a, f)
    return out


def tlr_gemm_workspace_bytes(h: int, opA: int, opB: int, A: tlr_operand_t, B: tlr_operand_t, runs: int) -> int:
    n = ctypes.c_size_t()
    check(lib().tlr_gemm_workspace_bytes(_P(h), opA, opB, ctypes.byref(A), ctypes.byref(B), runs,
                                         ctypes.byref(n)), "tlr_gemm_workspace_bytes")
    return n.value


def tlr_gemm_workspace_bytes_for_order(h: int, opA: int, opB: int, A: tlr_operand_t, B: tlr_operand_t, runs: int,
                                       order: int) -> int:
    n = ctypes.c_size_t()
    check(lib().tlr_gemm_workspace_bytes_for_order(_P(h), opA, opB, ctypes.byref(A), ctypes.byref(B), runs, order,
                                                   ctypes.byref(n)), "tlr_gemm_workspace_bytes_for_order")
    return n.value


def tlr_plan_create(h: int, opA: int, opB: int, A: tlr_operand_t, B: tlr_operand_t, ws: int, ws_bytes: int,
                    order: int = TLR_ORDER_AUTO) -> int:
    p = _P()
    check(lib().tlr_plan_create(_P(h), opA, opB, ctypes.byref(A), ctypes.byref(B), _P(ws), ws_bytes, order,
                                ctypes.byref(p)), "tlr_plan_create")
    return p.value


def _info_dict(i) -> dict:
    d = {f: getattr(i, f) for f, _ in tlr_plan_info_t._fields_}
    d["flops_launch"] = list(i.flops_launch)
    return d


def tlr_plan_info(p: int) -> dict:
    i = tlr_plan_info_t()
    check(lib().tlr_plan_info(_P(p), ctypes.byref(i)), "tlr_plan_info")
    return _info_dict(i)


def _rects(call, what: str) -> list:
    n = ctypes.c_int32()
    check(call(None, 0, ctypes.byref(n)), what)
    arr = (tlr_rect_t * max(1, n.value))()
    check(call(arr, n.value, ctypes.byref(n)), what)
    names = {TLR_ORDER_RIGHT: "R", TLR_ORDER_LEFT: "L", TLR_ORDER_TRIPLE: "P"}
    return [(r.i0, r.i1, r.j0, r.j1, names.get(r.order, r.order)) for r in arr[:n.value]]


def tlr_plan_rects(p: int) -> list:
    """[(i0, i1, j0, j1, order)] of a plan, order "R", "L" or "P" (per tile triple)."""
    return _rects(lambda a, c, n: lib().tlr_plan_rects(_P(p), a, c, n), "tlr_plan_rects")


def tlr_debug_plan_rects(opA: int, opB: int, A: tlr_operand_t, B: tlr_operand_t, ws_bytes: int,
                         order: int = TLR_ORDER_AUTO) -> list:
    """The rectangles a plan for this budget would use (host only, no device)."""
    return _rects(lambda a, c, n: lib().tlr_debug_plan_rects(opA, opB, ctypes.byref(A), ctypes.byref(B), ws_bytes,
                                                             order, a, c, n), "tlr_debug_plan_rects")


def tlr_plan_execute(p: int, alpha: float, beta: float, C: int, ldc: int) -> None:
    check(lib().tlr_plan_execute(_P(p), alpha, beta, _P(C), ldc), "tlr_plan_execute")


def tlr_plan_destroy(p: int) -> None:
    check(lib().tlr_plan_destroy(_P(p)), "tlr_plan_destroy")


def tlr_gemm(h: int, opA: int, opB: int, alpha: float, A: tlr_operand_t, B: tlr_operand_t, beta: float,
             C: int, ldc: int, ws: int, ws_bytes: int) -> None:
    check(lib().tlr_gemm(_P(h), opA, opB, alpha, ctypes.byref(A), ctypes.byref(B), beta, _P(C), ldc,
                         _P(ws), ws_bytes), "tlr_gemm")


def tlr_gemm_static_scratch(h: int, opA: int, opB: int, alpha: float, A: tlr_operand_t, B: tlr_operand_t,
                            beta: float, C: int, ldc: int) -> None:
    check(lib().tlr_gemm_static_scratch(_P(h), opA, opB, alpha, ctypes.byref(A), ctypes.byref(B), beta, _P(C),
                                        ldc), "tlr_gemm_static_scratch")


def tlr_get_device_status(h: int) -> int:
    return lib().tlr_get_device_status(_P(h))


def tlr_set_timing(h: int, enabled: bool) -> None:
    check(lib().tlr_set_timing(_P(h), 1 if enabled else 0), "tlr_set_timing")


def tlr_get_timing(h: int, kind: int):
    ms, n = ctypes.c_double(), ctypes.c_int64()
    check(lib().tlr_get_timing(_P(h), kind, ctypes.byref(ms), ctypes.byref(n)), "tlr_get_timing")
    return ms.value, n.value


def tlr_reset_timing(h: int) -> None:
    check(lib().tlr_reset_timing(_P(h)), "tlr_reset_timing")


def tlr_set_wait_limit_us(h: int, us: int) -> None:
    check(lib().tlr_set_wait_limit_us(_P(h), us), "tlr_set_wait_limit_us")


def tlr_debug_unsatisfied_wait(h: int) -> None:
    check(lib().tlr_debug_unsatisfied_wait(_P(h)), "tlr_debug_unsatisfied_wait")


def tlr_debug_check_plan(opA: int, opB: int, A: tlr_operand_t, B: tlr_operand_t, ws_bytes: int,
                         order: int = TLR_ORDER_AUTO):
    """(status, reason, plan info) of the host-side table check; no device use."""
    info = tlr_plan_info_t()
    msg = ctypes.create_string_buffer(512)
    st = lib().tlr_debug_check_plan(opA, opB, ctypes.byref(A), ctypes.byref(B), ws_bytes, order,
                                    ctypes.byref(info), msg, 512)
    return st, msg.value.decode(), _info_dict(info)


def tlr_compress_workspace_bytes(b: int, s: int, tiles: int) -> int:
    n = ctypes.c_size_t()
    check(lib().tlr_compress_workspace_bytes(b, s, tiles, ctypes.byref(n)), "tlr_compress_workspace_bytes")
    return n.value


def tlr_compress(h: int, C: int, ldc: int, m: int, n: int, b: int, dense_diagonal: bool, eps: float, r_max: int,
                 omega: int, s: int, U: int, V: int, D: int, ranks: int, errors: int, ws: int, ws_bytes: int) -> None:
    check(lib().tlr_compress(_P(h), _P(C), ldc, m, n, b, 1 if dense_diagonal else 0, eps, r_max, _P(omega), s,
                             _P(U), _P(V), _P(D), _P(ranks), _P(errors), _P(ws), ws_bytes), "tlr_compress")


def tlr_pack(h: int, n: int, b: int, r_max: int, ranks_host, U_pad: int, V_pad: int, D_pad: int, U: int, V: int,
             D: int, bu_U: int, bu_V: int, bv_U: int, bv_V: int, gamma: int) -> None:
    """ranks_host: a C-contiguous int32 numpy array of the nt x nt ranks."""
    import numpy as np
    r = np.ascontiguousarray(ranks_host, dtype=np.int32)
    check(lib().tlr_pack(_P(h), n, b, r_max, _P(r.ctypes.data), _P(U_pad), _P(V_pad), _P(D_pad), _P(U), _P(V),
                         _P(D), _P(bu_U), _P(bu_V), _P(bv_U), _P(bv_V), _P(gamma)), "tlr_pack")
