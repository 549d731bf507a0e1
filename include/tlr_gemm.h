/*
 * tlr_gemm.h -- C ABI of the GB300 (sm_103a) Tile-Low-Rank GEMM library.
 *
 * Operation ("Tile-Low-Rank GEMM: Designing Storage Around the Contraction",
 * opening section):   C <- alpha * op(A) * op(B) + beta * C
 * with C dense (fp32, column-major) and one or both of A, B in TLR format.
 *
 * TLR format (same page, sections "Many small GEMMs" and "Packing for the
 * contraction"; "TLR Matrix Multiplication", section "Introduction: TLR GEMM"):
 *   - an nt_r x nt_c grid of tiles, interior tiles b x b; a square matrix whose
 *     order N is not a multiple of b has a last tile row/column of
 *     b_rem = N - m*b (m = N / b);
 *   - with diag_dense != 0 the diagonal tiles are dense, every other tile
 *     (i,k) is U_ik V_ik^T with its own rank r_ik (0 <= r_ik <= min(d_i, d_k));
 *   - outer factors U are packed by tile row (i ascending, then k ascending),
 *     inner factors V by tile column (k ascending, then i ascending); dense tiles
 *     are skipped; every factor is column-major with leading dimension equal to
 *     its own dense dimension (d_i for U_ik, d_k for V_ik) and takes exactly
 *     r_ik columns (no padding); each tile's place follows from a prefix sum
 *     of the ranks;
 *   - dense diagonal tiles: a b x b x m array, tile i column-major at i*b*b;
 *   - boundary panels ("TLR Matrix Multiplication", section "Introduction:
 *     TLR GEMM"): when N % b != 0 the interior m x m grid lives in U, V, D and
 *     the boundary column u (tiles (i,m), i < m), the boundary row v^T (tiles
 *     (m,j), j < m) and the dense b_rem x b_rem corner gamma have buffers of
 *     their own: bu_U (b x r_im factors) and bu_V (b_rem x r_im) packed by
 *     ascending i; bv_U (b_rem x r_mj) and bv_V (b x r_mj) packed by ascending
 *     j; gamma column-major with leading dimension b_rem.
 *   Boundary panels are defined for square TLR matrices with a dense diagonal;
 *   a TLR matrix without dense diagonal (all tiles low-rank, e.g. the worked
 *   example's 2x3 grid) may be rectangular but its dimensions must be
 *   multiples of b.
 *
 * Conventions for every entry point:
 *   - All numeric buffers are DEVICE pointers owned by the caller; the library
 *     never frees or reallocates them. Device means cudaMalloc or managed
 *     memory: a host pointer (pinned or not) for an operand, the workspace or C
 *     gets TLR_STATUS_INVALID_ARG before any table is built or kernel launched.
 *     Rank and offset arrays are HOST pointers, read during the call (a plan
 *     keeps its own copy).
 *   - Element types: fp32 (run on TF32 tensor cores, inputs rounded to nearest
 *     TF32 first), bf16 or fp16 (tensor cores, fp32 accumulation; the
 *     intermediate S, T and P products are kept in the input type, rounded to
 *     nearest even). Both operands of one product have the same element type.
 *     C is always fp32.
 *   - Alignment: every base pointer 16-byte aligned; every leading dimension
 *     (and each tile's dense dimension) times the element size a multiple of 16
 *     bytes (d % 4 == 0 for fp32, d % 8 == 0 for bf16 and fp16); ldc % 4 == 0.
 *     Violations return TLR_STATUS_ALIGNMENT before anything is launched.
 *   - Calls are asynchronous on the handle's stream (BLAS convention). A
 *     status other than TLR_STATUS_OK means nothing was launched, except
 *     TLR_STATUS_CUDA_ERROR from a failed launch.
 *   - beta == 0: C is not read (it may hold NaN). alpha == 0: the operands are
 *     not read and C <- beta * C.
 *   - Nothing throws across the ABI.
 */
#ifndef TLR_GEMM_H
#define TLR_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TLR_STATUS_OK = 0,
    TLR_STATUS_INVALID_ARG = 1,        /* bad dimension, rank, pointer or enum */
    TLR_STATUS_ALIGNMENT = 2,          /* pointer / leading dimension not 16-byte aligned */
    TLR_STATUS_WORKSPACE_TOO_SMALL = 3,/* budget below the minimum one rectangle needs */
    TLR_STATUS_UNSUPPORTED = 4,        /* valid but not provided (e.g. dense x dense) */
    TLR_STATUS_CUDA_ERROR = 5,         /* a CUDA runtime call or launch failed */
    TLR_STATUS_TIMEOUT = 6,            /* a device-side wait ran out (kernel returned early) */
    TLR_STATUS_NOT_INITIALIZED = 7     /* no CUDA device, or the handle is unusable */
} tlr_status_t;

typedef enum { TLR_OP_N = 0, TLR_OP_T = 1 } tlr_op_t;
typedef enum { TLR_F32 = 0, TLR_BF16 = 1, TLR_F16 = 2 } tlr_dtype_t;
typedef enum { TLR_KIND_TLR = 0, TLR_KIND_DENSE = 1 } tlr_kind_t;
/* Association order of the low-rank products (page 1, "Association order and
 * workspace"; page 2, "The O_A O_B terms"): RIGHT U (S Z^T) or LEFT (U S) Z^T
 * everywhere; PER_RECT the cheaper of the two per output rectangle; TRIPLE
 * decided per tile triple (i, k, j) by min(r_ik, r_kj) after S_ikj = V_ik^T W_kj
 * (two TLR operands with a 16-bit element type; otherwise
 * TLR_STATUS_UNSUPPORTED). AUTO takes TRIPLE where it is available and its
 * final stage needs at most 90 % of the FLOPs of the cheaper single order over
 * all of C, else PER_RECT. */
typedef enum {
    TLR_ORDER_AUTO = 0, TLR_ORDER_RIGHT = 1, TLR_ORDER_LEFT = 2, TLR_ORDER_TRIPLE = 3, TLR_ORDER_PER_RECT = 4
} tlr_order_t;

/* One operand. Fields not used by its kind must be zero / NULL. */
typedef struct tlr_operand {
    int32_t kind;            /* tlr_kind_t */
    int32_t dtype;           /* tlr_dtype_t */
    int64_t rows, cols;      /* dimensions of the stored matrix (before op) */
    /* ---- TLR ---- */
    int32_t b;               /* nominal tile size */
    int32_t diag_dense;      /* 1: diagonal tiles dense (square only) */
    const int32_t *ranks;    /* HOST, nt_r * nt_c row-major; diagonal entries ignored when diag_dense */
    const int64_t *u_offsets;/* HOST, optional (NULL): element offset of each low-rank tile's outer
                                factor in its buffer (U, bu_U or bv_U), nt_r*nt_c row-major; checked
                                against the prefix sums of the ranks */
    const int64_t *v_offsets;/* HOST, optional: same for the inner factor (V, bu_V or bv_V) */
    const void *U, *V;       /* DEVICE, packed interior factors */
    const void *D;           /* DEVICE, dense diagonal tiles (b*b*m), or NULL without dense diagonal */
    const void *bu_U, *bu_V; /* DEVICE, boundary column factors (NULL when N % b == 0) */
    const void *bv_U, *bv_V; /* DEVICE, boundary row factors */
    const void *gamma;       /* DEVICE, dense boundary corner */
    /* ---- DENSE ---- */
    const void *data;        /* DEVICE, column-major */
    int64_t ld;              /* leading dimension (>= rows) */
} tlr_operand_t;

typedef struct tlr_handle_s *tlr_handle_t;
typedef struct tlr_plan_s *tlr_plan_t;

/* Summary of a plan (all FLOP counts at logical ranks, 2*M*N*K per product). */
typedef struct tlr_plan_info {
    int32_t runs;                 /* output rectangles executed in sequence */
    int32_t runs_right, runs_left;/* rectangles using each association order */
    int32_t runs_triple;          /* rectangles with the order chosen per tile triple */
    int64_t launches;             /* kernel launches per execution */
    double flops_executed;        /* every product the plan runs */
    double flops_stage1, flops_stage2, flops_stage3, flops_dense_terms;
    double flops_right_final, flops_left_final;  /* F_R and F_L summed over the rectangles */
    size_t workspace_bytes;       /* bytes of the caller's workspace the plan uses */
    int64_t tasks;                /* output tiles over all launches */
    double flops_launch[3];       /* per execution, by launch class: [0] Stage 1 with the
                                     dense-tile precomputes, [1] Stage 2, [2] Stage 3 */
} tlr_plan_info_t;

/* One output rectangle of a plan: tile rows [i0, i1) and tile columns [j0, j1)
 * of C's tile grid, evaluated with association order `order` (tlr_order_t:
 * TLR_ORDER_RIGHT U (S Z^T), TLR_ORDER_LEFT (U S) Z^T (page 1, "Association
 * order and workspace"), or TLR_ORDER_TRIPLE, the order taken per tile triple
 * (page 2, "The O_A O_B terms")). Rectangles run in the order listed. */
typedef struct tlr_rect {
    int32_t i0, i1, j0, j1;
    int32_t order;
} tlr_rect_t;

/* Metadata of a TLR x TLR product computed from ranks alone (no device use).
 * Arrays are caller-owned with the stated lengths. */
typedef struct tlr_analysis {
    int32_t nt_i, nt_k, nt_j;     /* tile grid of op(A) rows, contraction, op(B) columns */
    int64_t *rho;                 /* [nt_i] rank sums of op(A)'s tile rows (low-rank tiles) */
    int64_t *gamma;               /* [nt_j] rank sums of op(B)'s tile columns */
    int64_t *sigma;               /* [nt_k] rank sums of op(A)'s tile columns */
    int64_t *Gamma;               /* [nt_k] rank sums of op(B)'s tile rows */
    int64_t *stage1_mnk;          /* [3*nt_k] Stage-1 product shape per k */
    int64_t *stage3_mnk;          /* [3*nt_i] Stage-3 product shape per tile row (right order, all of C) */
    double F_R, F_L;              /* final-stage costs of the two orders over all of C */
    int32_t order;                /* TLR_ORDER_RIGHT or TLR_ORDER_LEFT (tie: right) */
    int64_t T_right_rows, T_right_cols, T_left_rows, T_left_cols; /* terminal workspaces (elements) */
    int64_t coupling_products;    /* (i,k,j) with both tiles low-rank and non-zero rank */
    int64_t distinct_shapes;      /* distinct (r_ik, r_kj) among them */
    double F_P;                   /* final-stage cost of the per-triple order over all of C on the
                                     terms of F_R and F_L (page 2, "The O_A O_B terms": K = min(r_ik,
                                     r_kj) per low-rank triple, K = r_ij for the k = j block) */
} tlr_analysis_t;

/* Status name, never NULL. */
const char *tlr_status_string(tlr_status_t s);

/* Create a handle on the current CUDA device. `stream` is a cudaStream_t
 * (NULL: the legacy default stream). The handle owns an error word in device
 * memory and (when timing is on) CUDA events; it owns no caller buffer. */
tlr_status_t tlr_create(tlr_handle_t *handle, void *stream);
tlr_status_t tlr_destroy(tlr_handle_t handle);
tlr_status_t tlr_set_stream(tlr_handle_t handle, void *stream);

/* Rank metadata of op(A) * op(B) for two TLR descriptors; host only, no
 * pointer fields are read (page 1, "Association order and workspace"). */
tlr_status_t tlr_analyze(tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A,
                         const tlr_operand_t *B, tlr_analysis_t *out);

/* Workspace needed so that the planner splits C into at most `runs`
 * rectangles (page 1, "Association order and workspace": the budget for a
 * target number of runs). runs <= 0 means one run. */
tlr_status_t tlr_gemm_workspace_bytes(tlr_handle_t handle, tlr_op_t opA, tlr_op_t opB,
                                      const tlr_operand_t *A, const tlr_operand_t *B,
                                      int runs, size_t *bytes);
/* The same for a plan created with association order `order` (the call above
 * sizes for TLR_ORDER_AUTO); TLR_STATUS_UNSUPPORTED where the order cannot apply. */
tlr_status_t tlr_gemm_workspace_bytes_for_order(tlr_handle_t handle, tlr_op_t opA, tlr_op_t opB,
                                                const tlr_operand_t *A, const tlr_operand_t *B,
                                                int runs, tlr_order_t order, size_t *bytes);

/* Plan a product: validate the descriptors, compute the rank prefixes, split C
 * into rectangles of output tiles that fit `workspace_bytes`, choose the
 * association order (`order`, see tlr_order_t), and build the
 * device-side descriptor tables. The plan binds the operand buffers and the
 * workspace pointer (caller-owned, >= workspace_bytes, 256-byte aligned); it
 * owns only its small descriptor tables. */
tlr_status_t tlr_plan_create(tlr_handle_t handle, tlr_op_t opA, tlr_op_t opB,
                             const tlr_operand_t *A, const tlr_operand_t *B,
                             void *workspace, size_t workspace_bytes,
                             tlr_order_t order, tlr_plan_t *plan);
tlr_status_t tlr_plan_info(tlr_plan_t plan, tlr_plan_info_t *info);
/* The plan's output rectangles (host copy): at most `capacity` are written to
 * `rects` (caller-owned; NULL when capacity is 0) and *count receives how many
 * the plan has, so a first call with capacity 0 sizes the array. Lets a
 * caller recount the plan's executed FLOPs from the ranks on its own. */
tlr_status_t tlr_plan_rects(tlr_plan_t plan, tlr_rect_t *rects, int32_t capacity, int32_t *count);
/* Run a planned product into C (device, fp32, column-major, leading dimension ldc). */
tlr_status_t tlr_plan_execute(tlr_plan_t plan, float alpha, float beta, float *C, int64_t ldc);
tlr_status_t tlr_plan_destroy(tlr_plan_t plan);

/* One-shot product (plan, execute, release). The plan's descriptor tables are
 * freed after the stream has drained them. */
tlr_status_t tlr_gemm(tlr_handle_t handle, tlr_op_t opA, tlr_op_t opB, float alpha,
                      const tlr_operand_t *A, const tlr_operand_t *B, float beta,
                      float *C, int64_t ldc, void *workspace, size_t workspace_bytes);

/* Size of the static device scratch used by tlr_gemm_static_scratch: 64 MiB. */
#define TLR_STATIC_SCRATCH_BYTES ((size_t)64 * 1024 * 1024)

/* One-shot product like tlr_gemm, but with no workspace argument and no device
 * allocation: the workspace, descriptor tables and counters live in one static
 * device array of TLR_STATIC_SCRATCH_BYTES inside the library, reserved by the
 * CUDA runtime when it loads the module that holds the array (with lazy module
 * loading, during the first call on a device). The method's description has no
 * counterpart to this call; it serves callers that may not allocate device
 * memory while they run (an allocator that owns all free memory, or a loop
 * that must not stall on allocation).
 *   Setup: the first call on each device (that device current) looks up the
 *   array's device address with cudaGetSymbolAddress and keeps it. After the
 *   device's context has been destroyed and re-created (cudaDeviceReset), the
 *   next call looks the address up again. The current device must be the
 *   handle's device (the one current at tlr_create), else
 *   TLR_STATUS_INVALID_ARG.
 *   Sharing: every call on a device, from any handle or thread, uses the same
 *   array. Calls must be ordered (one stream, or events between streams);
 *   overlapping calls race on the workspace and the counters and give wrong
 *   results. The counters are zeroed on the stream at every call; nothing else
 *   needs to start at zero.
 *   Limits: the planner splits C into rectangles to fit the array; a product
 *   whose smallest split, plus its tables, exceeds it returns
 *   TLR_STATUS_WORKSPACE_TOO_SMALL before anything is launched or copied.
 *   Host memory is used for planning as in every other call; with timing on,
 *   the handle may create CUDA events. Other errors as tlr_gemm. */
tlr_status_t tlr_gemm_static_scratch(tlr_handle_t handle, tlr_op_t opA, tlr_op_t opB, float alpha,
                                     const tlr_operand_t *A, const tlr_operand_t *B, float beta,
                                     float *C, int64_t ldc);

/* Asynchronous device status: synchronises the handle's stream and returns
 * TLR_STATUS_TIMEOUT if a kernel ran out of a bounded wait since the last call
 * (the word is then cleared), TLR_STATUS_CUDA_ERROR on a sticky CUDA error. */
tlr_status_t tlr_get_device_status(tlr_handle_t handle);

/* Per-kernel timing with CUDA events on the handle's stream. While enabled,
 * every launch is bracketed by an event pair; tlr_get_timing synchronises and
 * returns, for launch class `kind`, the summed milliseconds and launch count
 * since the last reset. Classes: 1 the launch of a rectangle's Stages 1-2 and
 * dense precomputes, 2 the launch of its final products (products whose final
 * tiles run on CTA pairs use these two launches per rectangle); 5 a whole
 * product in one launch (every other product); 3 the fp32 rounding and
 * transpose pre-pass; 4 the alpha == 0 scale-only kernel; 0 Stage 1 and the
 * dense precomputes in a launch of their own (products with a dense operand,
 * where they run on CTA pairs before the final products; also the per-stage
 * diagnostic schedule, which then leaves Stage 2 alone in class 1). */
tlr_status_t tlr_set_timing(tlr_handle_t handle, int enabled);
tlr_status_t tlr_get_timing(tlr_handle_t handle, int kind, double *ms, int64_t *launches);
tlr_status_t tlr_reset_timing(tlr_handle_t handle);

/* ---- TLR output ("TLR Matrix Multiplication", section "Introduction: TLR
 * GEMM": the TLR-output cases of the product). A TLR-output product is the
 * dense-output product (tlr_gemm into a dense scratch C, which holds
 * beta * C0 on entry) followed by tlr_compress of that C, and tlr_pack to the
 * packed TLR format of this header. Neither page describes the recompression;
 * the rule here is the truncated SVD of each tile:
 *   every tile (i, j) of C's grid (b x b, the last row/column of tiles
 *   ragged) except the diagonal ones when dense_diagonal != 0 (square C) gets
 *   the smallest rank r with sqrt(sum_{k > r} sigma_k^2) <= eps * ||C_ij||_F,
 *   capped at min(r_max, d_i, d_j); U_ij V_ij^T approximates C_ij.
 * Method (per tile, fp32 arithmetic, tile energies in fp64): sketch
 * Y = C_ij Omega with the caller's s columns of Omega (b x s, column-major,
 * leading dimension b; typically Gaussian; random numbers are an input),
 * orthonormal basis Q of Y (Gram-Schmidt with reorthogonalisation),
 * B = Q^T C_ij, Jacobi eigen-decomposition of B B^T, then the rule above on
 * ||C_ij||^2 minus the kept eigenvalues, U = Q W_r (orthonormal columns),
 * V = B^T W_r. With s above a tile's numerical rank the result is that tile's
 * truncated SVD up to rounding; otherwise the rank can exceed the optimal one
 * and the rule still bounds the error, which is returned per tile. Energies
 * are resolved to about 1e-5 of a tile's, so eps below about 3e-3 decides ranks
 * on rounding.
 *
 * tlr_compress arguments (DEVICE pointers unless stated):
 *   C (m x n, column-major, ldc >= m) is read only; b tile size; s even,
 *   2 <= s <= 128; 0 <= r_max <= s; eps >= 0.
 *   Outputs, tile t = i * nJ + j of the nI x nJ grid (nI = ceil(m/b)):
 *   ranks[t] (int32) and errors[t] (relative Frobenius error of U V^T; 0 for
 *   dense tiles); U: a b x r_max column-major block per tile at t*b*r_max
 *   (leading dimension b, rows d_i used, columns from ranks[t] on zero); V
 *   likewise with rows d_j; D (dense_diagonal only): diagonal tile t at t*b*b,
 *   leading dimension b. U and V may be NULL when r_max == 0.
 *   workspace: at least tlr_compress_workspace_bytes(b, s, 1); with more, up
 *   to tlr_compress_workspace_bytes(b, s, nI*nJ), more tiles run at once.
 *   Asynchronous on the handle's stream; the current device must be the
 *   handle's. Errors: TLR_STATUS_INVALID_ARG (bad size, argument or host
 *   pointer), TLR_STATUS_WORKSPACE_TOO_SMALL, TLR_STATUS_UNSUPPORTED (b above
 *   what one block's shared memory holds), TLR_STATUS_CUDA_ERROR. */
tlr_status_t tlr_compress_workspace_bytes(int64_t b, int32_t s, int64_t tiles, size_t *bytes);
tlr_status_t tlr_compress(tlr_handle_t handle, const float *C, int64_t ldc, int64_t m, int64_t n, int64_t b,
                          int32_t dense_diagonal, float eps, int32_t r_max, const float *omega, int32_t s,
                          float *U, float *V, float *D, int32_t *ranks, float *errors, void *workspace,
                          size_t workspace_bytes);

/* Packs the output of tlr_compress for a square n x n matrix with dense
 * diagonal into the fp32 TLR buffers that a tlr_operand_t points at: interior
 * U by tile row, V by tile column, D; with n % b != 0 also the boundary panels
 * bu_U, bu_V, bv_U, bv_V and the corner gamma. `ranks` is a HOST copy of tlr_compress's ranks
 * (nt * nt, nt = ceil(n/b); 0 on the diagonal). Each destination holds exactly
 * the prefix-summed sizes of this header's format; buffers for parts with no
 * columns may be NULL. Asynchronous on the handle's stream. */
tlr_status_t tlr_pack(tlr_handle_t handle, int64_t n, int64_t b, int32_t r_max, const int32_t *ranks,
                      const float *U_pad, const float *V_pad, const float *D_pad, float *U, float *V, float *D,
                      float *bu_U, float *bu_V, float *bv_U, float *bv_V, float *gamma);

/* Host-only check of the tables a plan would launch, with no device use.
 * Pointer fields of A and B may be arbitrary distinct 16-byte-aligned values
 * (nothing is dereferenced). Builds the plan for `workspace_bytes` and
 * verifies that every TMA view lies inside an input buffer or the workspace,
 * every task writes inside its output, C is covered exactly once and every
 * terminal-matrix row Stage 3 reads is written exactly once. On failure returns
 * TLR_STATUS_INVALID_ARG with a reason in msg. */
tlr_status_t tlr_debug_check_plan(tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A,
                                  const tlr_operand_t *B, size_t workspace_bytes, tlr_order_t order,
                                  tlr_plan_info_t *info, char *msg, size_t msg_len);

/* Host-only: the rectangles tlr_plan_create would choose for these operands,
 * budget and order (same split, same per-rectangle order), without device use;
 * pointer fields of A and B are not read. Array protocol as tlr_plan_rects. */
tlr_status_t tlr_debug_plan_rects(tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A,
                                  const tlr_operand_t *B, size_t workspace_bytes, tlr_order_t order,
                                  tlr_rect_t *rects, int32_t capacity, int32_t *count);

/* Test hook: device wait limit in microseconds for this handle's kernels
 * (default 2,000,000). Used by the bounded-wait test, which gives a kernel a
 * wait that nothing satisfies and checks TLR_STATUS_TIMEOUT comes back. */
tlr_status_t tlr_set_wait_limit_us(tlr_handle_t handle, int64_t limit_us);
tlr_status_t tlr_debug_unsatisfied_wait(tlr_handle_t handle);

#ifdef __cplusplus
}
#endif
#endif /* TLR_GEMM_H */
