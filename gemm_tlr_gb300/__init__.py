"""GB300 (sm_103a) Tile-Low-Rank GEMM: C <- alpha op(A) op(B) + beta C.

The compute path is ``libtlrgemm.so`` (hand-written tcgen05/TMA/TMEM kernels and
a native planner) behind the C ABI of ``include/tlr_gemm.h``. This package is a
thin binding: ``_abi`` mirrors the C entry points one to one, ``device`` moves
seeded host inputs into device memory with PyTorch (memory and streams only)
and builds the operand descriptors, and ``flops`` counts executed FLOPs from
ranks for the benchmark's metric.
"""
from ._abi import (  # noqa: F401
    TLR_BF16, TLR_F16, TLR_F32, TLR_KIND_DENSE, TLR_KIND_TLR, TLR_OP_N, TLR_OP_T, TLR_ORDER_AUTO,
    TLR_ORDER_LEFT, TLR_ORDER_PER_RECT, TLR_ORDER_RIGHT, TLR_ORDER_TRIPLE, TLRError, header_symbols, lib, tlr_analysis_t,
    tlr_analyze, tlr_compress, tlr_compress_workspace_bytes, tlr_create, tlr_debug_check_plan, tlr_debug_plan_rects, tlr_debug_unsatisfied_wait, tlr_destroy, tlr_gemm,
    tlr_gemm_static_scratch, tlr_gemm_workspace_bytes, tlr_gemm_workspace_bytes_for_order, tlr_get_device_status, tlr_get_timing, tlr_operand_t,
    tlr_pack, tlr_plan_create, tlr_plan_destroy, tlr_plan_execute, tlr_plan_info, tlr_plan_rects, tlr_rect_t,
    tlr_reset_timing,
    tlr_set_stream, tlr_set_timing, tlr_set_wait_limit_us, tlr_status_string,
)
