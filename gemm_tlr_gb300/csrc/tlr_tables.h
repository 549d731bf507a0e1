// Device-side descriptor tables shared by the host planner (tlr_plan.cu) and
// the tcgen05 kernel (tlr_kernels.cu). Everything here is plain data: the
// planner fills these arrays once per plan and uploads them; each kernel launch
// walks a contiguous range of tasks.
//
// A task is one 128 x BN output tile of one product. Its accumulator is the
// sum over a short list of K segments; each segment is one operand pair read
// through two TMA tensor maps with exact extents (so ragged ranks are
// zero-filled by the copy engine, never padded in memory). This is how the sum
// over contraction tiles k runs inside one tensor-core K-loop ("Tile-Low-Rank
// GEMM: Designing Storage Around the Contraction", section "One product, three
// stages", Stage 3) and how the dense-diagonal terms of "TLR Matrix
// Multiplication", section "Regular TLR GEMM", join the same accumulator so C is
// written once.
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace tlr {

constexpr int kBM = 128;            // rows of an output tile (MMA M)
constexpr int kMaxBN = 256;         // widest output tile (MMA N)
constexpr int kStages = 4;          // shared-memory pipeline depth
constexpr int kSmemA = kBM * 128;   // one stage of A: 128 rows x 128 bytes
constexpr int kSmemB = kMaxBN * 128;
constexpr int kStageBytes = kSmemA + kSmemB;
#ifndef TLR_EPI_GROUPS
#define TLR_EPI_GROUPS 2
#endif
constexpr int kEpiGroups = TLR_EPI_GROUPS;   // epilogue warp groups; each stores every kEpiGroups-th 64-column block
constexpr int kEpiThreads = 128 * kEpiGroups;
constexpr int kThreads = 96 + kEpiThreads;   // warp 0 TMA, warp 1 MMA, warp 2 descriptors, then the epilogue
constexpr int kTmemCols = 512;      // two accumulators of up to 256 fp32 columns, or four of 128
constexpr int kMaxAcc = 4;          // accumulators in TMEM at most (tiles at most 128 wide)
constexpr int kMaxSegs = 8;         // K segments per task
constexpr int kRing = 8;            // task descriptors staged ahead in shared memory
constexpr int kTicketBatch = 4;     // consecutive tickets a CTA (or CTA pair) claims at once
constexpr int kSlotBytes = 1536;    // one staged task: header, segments, per-row destinations
constexpr int kEpiStageBytes = 2048; // per epilogue warp: a 32 x 32 bf16 block on its way to a row-major output
constexpr int kSignalBatch = 16;    // completion signals an epilogue warp may hold back (same counter)
constexpr int kSmemBytes = kStages * kStageBytes + kRing * kSlotBytes + 1024 /*align*/ + 512 /*barriers*/ +
                           4 * kEpiGroups * kEpiStageBytes;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(8 * (2 * kStages + 2 * kMaxAcc + 2 + 2 * kRing) + 16 <= 512, "barrier area");

enum : uint32_t {
  kSegAMN = 1u,   // A operand MN-major (rows of its view are M); else K-major
  kSegBMN = 2u,   // B operand MN-major (rows of its view are N); else K-major
};

// One K segment of a task. TMA coordinates are those of the first box; the
// kernel steps x/y by the box size along MN and by BK along K.
struct alignas(16) Seg {
  int32_t a_map, b_map;   // indices into the tensor-map table
  int32_t a_x, a_y;       // MN-major: (mn0, k0); K-major: (k0, mn0)
  int32_t b_x, b_y;
  int32_t k_len;          // logical K of this segment (elements, > 0)
  uint32_t flags;
};

// Row pieces: output-tile rows [src0, src0+len) go to output rows dst0.. .
struct alignas(16) Piece {
  int32_t src0, len;
  int64_t dst0;
};

enum : int32_t {
  kOutC = 0,        // fp32 C: alpha * acc + beta * C (C unread when beta == 0)
  kOutBF16 = 1,     // workspace, bf16 round-to-nearest-even
  kOutTF32 = 2,     // workspace, fp32 rounded to nearest tf32
  kOutF16 = 3,      // workspace, fp16 round-to-nearest-even
};

struct alignas(16) Out {
  void *ptr;        // NULL for kOutC: the launch's C pointer is used
  int64_t ld;       // ignored for kOutC (the launch's ldc)
  int32_t kind;
  int32_t trans;    // 1: element (r, c) of the tile goes to ptr[c + r * ld]
};

// Tasks of one launch are claimed in ticket order. A task may wait for up to
// two dependency counters to reach their targets before it starts (every
// counted task has a lower ticket, so the wait always ends) and signals one
// counter when done: each epilogue warp of each CTA working on the task adds
// one, so a counter's target is tasks x epilogue warps x CTAs per task. When
// `signal_writes` is set the increment is ordered after the warp's global
// stores (they are read later by TMA in other CTAs); otherwise it only records
// that the task's operand reads have finished.
struct alignas(16) Task {
  int32_t seg0, nseg;     // segments [seg0, seg0 + nseg); nseg == 0 writes zeros (beta * C)
  int32_t out;            // index into the output table
  int32_t rows, cols;     // valid part of the tile (<= kBM, <= BN)
  int32_t piece0, npiece; // row pieces; npiece == 0: output row = row0 + r
  int32_t signal;         // counter to increment when done, -1: none
  int64_t row0, col0;     // output coordinates of the tile origin
  int32_t dep[2];         // counters to wait for, -1: none
  uint32_t dep_target[2];
  int32_t signal_writes;  // 1: the increment publishes this task's stores
  int32_t pad_[3];
};

// One transposed input copy for the TF32 path: dst[c + r * dst_ld] =
// round_tf32(src[r + c * src_ld]) for r < rows, c < cols; tile0 is the first
// 32 x 32 tile of this job in the launch's tile numbering.
struct alignas(16) TJob {
  const float *src;
  float *dst;
  int64_t src_ld, dst_ld, rows, cols, tile0;
  int64_t pad_;
};

struct Params {
  // C as a 2-D fp32 tensor (rows x columns, column-major) for tensor-memory-
  // accelerated stores of whole 2 KiB blocks: [0] boxes of 32 rows x 16 columns,
  // [1] 16 rows x 32 columns with the 64-byte swizzle (transposed tiles).
  // Used when cmap_ok is set and beta == 0.
  CUtensorMap cmap[2];
  int32_t cmap_ok;
  int32_t f16;            // 16-bit operands are fp16 (else bf16); the TF32 kernel ignores it
  const void *maps;       // CUtensorMap[], 64-byte aligned, device memory
  const Task *tasks;
  const Seg *segs;
  const Piece *pieces;
  const Out *outs;
  float *C;
  int64_t ldc;
  float alpha, beta;
  int32_t ntasks;
  int32_t bn;             // output tile width (multiple of 64, <= kMaxBN)
  unsigned int *err;      // device error word (bounded waits that ran out)
  unsigned long long wait_limit_ns;
  unsigned int *ticket;   // next unclaimed task of this launch (zeroed before the launch)
  unsigned int *counters; // dependency counters (zeroed before the launch)
};

}  // namespace tlr
