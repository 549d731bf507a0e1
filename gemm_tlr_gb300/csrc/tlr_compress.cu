// Recompression of a dense matrix into TLR form: the step the TLR-output
// products add after the dense-output product ("TLR Matrix Multiplication",
// section "Introduction: TLR GEMM", names the TLR-output cases; "Tile-Low-Rank
// GEMM: Designing Storage Around the Contraction", section "Many small GEMMs",
// gives the format: each tile of a regular grid compressed on its own, its
// rank following its own compressibility). Neither page describes the
// recompression; the rule taken here is the truncated singular value
// decomposition of every off-diagonal tile with the smallest rank r whose
// discarded part is at most eps times the tile's Frobenius norm, capped at
// r_max.
//
// Per tile T (d_i x d_j, fp32), all in fp32 with the energies in fp64:
//   1. ||T||_F^2;
//   2. Y = T Omega, a sketch with s columns (randomized range finder of Halko,
//      Martinsson and Tropp, 2011; Omega is an input, drawn by the caller);
//   3. Q = an orthonormal basis of Y, classical Gram-Schmidt with one
//      reorthogonalisation (Giraud, Langou and Rozloznik, 2005);
//   4. B = Q^T T (s x d_j) and the core G = B B^T (s x s, fp64 accumulation
//      across blocks of 512 products);
//   5. G = W diag(lambda) W^T by the cyclic Jacobi method (two-sided
//      rotations, round-robin pair order; Golub and Van Loan, "Matrix
//      Computations", section 8.5), eigenvalues sorted in decreasing order:
//      lambda_k are the squared singular values of B;
//   6. r = the smallest rank with ||T||^2 - sum_{k<r} lambda_k <= eps^2 ||T||^2
//      (the energy left out of U V^T below, including what the sketch missed),
//      at most min(r_max, d_i, d_j, s);
//   7. U = Q W_r (d_i x r, orthonormal columns) and V = B^T W_r (d_j x r), so
//      that U V^T = Q W_r W_r^T Q^T T.
// When the sketch holds the tile's range (s above its numerical rank) this is
// the truncated SVD up to rounding; otherwise the rank may exceed the optimal
// one and the error stays within eps (or is reported when r_max caps it).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "tlr_gemm.h"

namespace tlr {
// handle access (tlr_plan.cu)
cudaStream_t handle_stream(tlr_handle_t h);
bool handle_on_current_device(tlr_handle_t h);
bool is_device_pointer(const void *p);
}

namespace tlr_cmp {

constexpr int kMaxSketch = 128;   // columns of the sketch (the core fits in shared memory)
constexpr int kThreads = 256;      // the GEMM blocks
constexpr int kBigThreads = 1024;  // one block per tile: energy, Jacobi
constexpr int kWarps = kBigThreads / 32;
constexpr int kPairsPerWarp = (kMaxSketch / 2 + kWarps - 1) / kWarps;   // Jacobi pairs per warp
constexpr int kOrthThreads = 512;  // one block per tile: Gram-Schmidt

struct Geo {
  int64_t m, n, b;
  int32_t nI, nJ;
  int32_t dense_diag;
  int32_t s, r_max;
  float eps;
};

__device__ __forceinline__ int64_t tile_dim(int64_t total, int64_t b, int64_t t) {
  const int64_t d = total - t * b;
  return d < b ? d : b;
}

// Per-tile scratch of one batch: Y/Q (b x s, ld b), B (s x b, ld s), G (s x s),
// W sorted (s x s), eigenvalues (s), the tile energy (fp64).
struct Scratch {
  float *Q, *B, *G, *W, *lam;
  double *norm2;
  int64_t q_stride, b_stride, g_stride;   // elements per tile
};

__device__ __forceinline__ bool is_dense_tile(const Geo &g, int64_t i, int64_t j) {
  return g.dense_diag && i == j;
}

// ---------------------------------------------------------------- tile energy
__global__ void __launch_bounds__(kBigThreads) norm_kernel(const float *C, int64_t ldc, Geo g, int64_t t0, Scratch w) {
  const int64_t t = t0 + blockIdx.x;
  const int64_t i = t / g.nJ, j = t % g.nJ;
  const int64_t di = tile_dim(g.m, g.b, i), dj = tile_dim(g.n, g.b, j);
  double acc = 0.0;
  if (!is_dense_tile(g, i, j)) {
    const float *T = C + i * g.b + j * g.b * ldc;
    for (int64_t c0 = 0; c0 < dj; c0 += 16) {   // fp32 sums of up to 16 x (b / blockDim) squares, then fp64
      float part = 0.f;
      const int64_t c1 = c0 + 16 < dj ? c0 + 16 : dj;
      for (int64_t c = c0; c < c1; ++c)
        for (int64_t r = threadIdx.x; r < di; r += blockDim.x) {
          const float x = T[r + c * ldc];
          part = fmaf(x, x, part);
        }
      acc += part;
    }
  }
  __shared__ double red[32];
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) s += red[k];
    w.norm2[blockIdx.x] = s;
  }
}

// ---------------------------------------------------------------- batched SIMT GEMM
// out(r, c) = sum_k A(r, k) B(k, c) for one TM x TN block of one tile, K in
// steps of TK; each of the 256 threads holds TM/16 x TN/16 results, its
// columns in groups of four 64 apart (tx * 4 + 64 g + y), so that the float4
// reads of a row of B touch consecutive addresses. kAk / kBk: the operand's
// contiguous index is k (else r for A, c for B), which decides the loading
// order so that neighbouring threads read neighbouring addresses (TK = 32
// gives 128-byte runs along a k-contiguous operand). kWide: partial sums of
// 512 products in fp32 are added into fp64 accumulators.
constexpr int kTN = 64;
template <int TM, int TK, bool kAk, bool kBk, bool kWide, int TN = kTN, class LA, class LB, class ST>
__device__ __forceinline__ void gemm_block(int64_t M, int64_t N, int64_t K, int64_t m0, int64_t n0, LA la, LB lb,
                                           ST st) {
  constexpr int RM = TM / 16;          // rows per thread (4 or 8)
  constexpr int CN = TN / 16;          // columns per thread (4 or 8)
  static_assert(TM == 64 || TM == 128, "tile rows");
  static_assert(TN == 64 || TN == 128, "tile columns");
  static_assert(TK == 16 || TK == 32, "tile depth");
  __shared__ __align__(16) float As[TK][TM + 4];
  __shared__ __align__(16) float Bs[TK][TN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[RM][CN];
  double wacc[kWide ? RM : 1][kWide ? CN : 1];
#pragma unroll
  for (int a = 0; a < RM; ++a)
#pragma unroll
    for (int c = 0; c < CN; ++c) acc[a][c] = 0.f;
  if constexpr (kWide) {
#pragma unroll
    for (int a = 0; a < RM; ++a)
#pragma unroll
      for (int c = 0; c < CN; ++c) wacc[a][c] = 0.0;
  }
  for (int64_t k0 = 0; k0 < K; k0 += TK) {
#pragma unroll
    for (int q = 0; q < TM * TK / kThreads; ++q) {
      const int idx = tid + kThreads * q;
      const int r = kAk ? idx / TK : idx % TM, k = kAk ? idx % TK : idx / TM;
      const int64_t gr = m0 + r, gk = k0 + k;
      As[k][r] = gr < M && gk < K ? la(gr, gk) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < TK * TN / kThreads; ++q) {
      const int idx = tid + kThreads * q;
      const int c = kBk ? idx / TK : idx % TN, kb = kBk ? idx % TK : idx / TN;
      const int64_t gc = n0 + c, gkb = k0 + kb;
      Bs[kb][c] = gc < N && gkb < K ? lb(gkb, gc) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < TK; ++k) {
      float a[RM], bb[CN];
#pragma unroll
      for (int h = 0; h < RM / 4; ++h) {
        const float4 a4 = *reinterpret_cast<const float4 *>(&As[k][ty * RM + 4 * h]);
        a[4 * h] = a4.x; a[4 * h + 1] = a4.y; a[4 * h + 2] = a4.z; a[4 * h + 3] = a4.w;
      }
#pragma unroll
      for (int h = 0; h < CN / 4; ++h) {
        const float4 b4 = *reinterpret_cast<const float4 *>(&Bs[k][64 * h + tx * 4]);
        bb[4 * h] = b4.x; bb[4 * h + 1] = b4.y; bb[4 * h + 2] = b4.z; bb[4 * h + 3] = b4.w;
      }
#pragma unroll
      for (int x = 0; x < RM; ++x)
#pragma unroll
        for (int y = 0; y < CN; ++y) acc[x][y] = fmaf(a[x], bb[y], acc[x][y]);
    }
    if constexpr (kWide) {
      if ((k0 & 511) == 512 - TK || k0 + TK >= K) {
#pragma unroll
        for (int x = 0; x < RM; ++x)
#pragma unroll
          for (int y = 0; y < CN; ++y) { wacc[x][y] += acc[x][y]; acc[x][y] = 0.f; }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int x = 0; x < RM; ++x)
#pragma unroll
    for (int y = 0; y < CN; ++y) {
      const int64_t r = m0 + ty * RM + x, c = n0 + 64 * (y / 4) + tx * 4 + (y % 4);
      if (r < M && c < N) {
        if constexpr (kWide) st(r, c, static_cast<float>(wacc[x][y]));
        else st(r, c, acc[x][y]);
      }
    }
}

// rows of the GEMM blocks of each kernel
constexpr int kSketchTM = 128, kProjTM = 64, kCoreTM = 64, kFactorTM = 128;

// Y = T Omega (d_i x s); TN: the block's columns (128 for sketches wider than
// 64 columns, so that each block reads its rows of T once)
template <int TN>
__global__ void __launch_bounds__(kThreads) sketch_kernel(const float *C, int64_t ldc, const float *omega, Geo g,
                                                          int64_t t0, Scratch w) {
  const int64_t t = t0 + blockIdx.z;
  const int64_t i = t / g.nJ, j = t % g.nJ;
  if (is_dense_tile(g, i, j)) return;
  const int64_t di = tile_dim(g.m, g.b, i), dj = tile_dim(g.n, g.b, j);
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kSketchTM, n0 = static_cast<int64_t>(blockIdx.y) * TN;
  if (m0 >= di || n0 >= g.s) return;
  const float *T = C + i * g.b + j * g.b * ldc;
  float *Y = w.Q + blockIdx.z * w.q_stride;
  const int64_t b = g.b;
  gemm_block<kSketchTM, 16, false, true, false, TN>(
      di, g.s, dj, m0, n0, [&](int64_t r, int64_t k) { return T[r + k * ldc]; },
      [&](int64_t k, int64_t c) { return omega[k + c * b]; }, [&](int64_t r, int64_t c, float v) { Y[r + c * b] = v; });
}

// B = Q^T T (s x d_j, ld s)
__global__ void __launch_bounds__(kThreads) project_kernel(const float *C, int64_t ldc, Geo g, int64_t t0, Scratch w) {
  const int64_t t = t0 + blockIdx.z;
  const int64_t i = t / g.nJ, j = t % g.nJ;
  if (is_dense_tile(g, i, j)) return;
  const int64_t di = tile_dim(g.m, g.b, i), dj = tile_dim(g.n, g.b, j);
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kProjTM, n0 = static_cast<int64_t>(blockIdx.y) * kTN;
  if (m0 >= g.s || n0 >= dj) return;
  const float *T = C + i * g.b + j * g.b * ldc;
  const float *Q = w.Q + blockIdx.z * w.q_stride;
  float *B = w.B + blockIdx.z * w.b_stride;
  const int64_t b = g.b, s = g.s;
  gemm_block<kProjTM, 32, true, true, true>(
      g.s, dj, di, m0, n0, [&](int64_t r, int64_t k) { return Q[k + r * b]; },
      [&](int64_t k, int64_t c) { return T[k + c * ldc]; }, [&](int64_t r, int64_t c, float v) { B[r + c * s] = v; });
}

// G = B B^T (s x s)
__global__ void __launch_bounds__(kThreads) core_kernel(Geo g, int64_t t0, Scratch w) {
  const int64_t t = t0 + blockIdx.z;
  const int64_t i = t / g.nJ, j = t % g.nJ;
  if (is_dense_tile(g, i, j)) return;
  const int64_t dj = tile_dim(g.n, g.b, j);
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kCoreTM, n0 = static_cast<int64_t>(blockIdx.y) * kTN;
  const float *B = w.B + blockIdx.z * w.b_stride;
  float *G = w.G + blockIdx.z * w.g_stride;
  const int64_t s = g.s;
  gemm_block<kCoreTM, 16, false, false, true>(
      s, s, dj, m0, n0, [&](int64_t r, int64_t k) { return B[r + k * s]; },
      [&](int64_t k, int64_t c) { return B[c + k * s]; }, [&](int64_t r, int64_t c, float v) { G[r + c * s] = v; });
}

// U = Q W (d_i x r_max) and V = B^T W (d_j x r_max), W with its columns from
// the rank on set to zero; written at the tile's place in the padded outputs.
__global__ void __launch_bounds__(kThreads) factor_kernel(Geo g, int64_t t0, Scratch w, float *Uo, float *Vo,
                                                          int which) {
  const int64_t t = t0 + blockIdx.z;
  const int64_t i = t / g.nJ, j = t % g.nJ;
  if (is_dense_tile(g, i, j)) return;
  const int64_t di = tile_dim(g.m, g.b, i), dj = tile_dim(g.n, g.b, j);
  const int64_t rows = which == 0 ? di : dj;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kFactorTM, n0 = static_cast<int64_t>(blockIdx.y) * kTN;
  if (m0 >= rows || n0 >= g.r_max) return;
  const float *W = w.W + blockIdx.z * w.g_stride;
  const int64_t b = g.b, s = g.s;
  float *out = (which == 0 ? Uo : Vo) + t * b * g.r_max;
  auto st = [&](int64_t r, int64_t c, float v) { out[r + c * b] = v; };
  auto lw = [&](int64_t k, int64_t c) { return W[k + c * s]; };
  if (which == 0) {
    const float *Q = w.Q + blockIdx.z * w.q_stride;
    gemm_block<kFactorTM, 16, false, true, false>(di, g.r_max, s, m0, n0, [&](int64_t r, int64_t k) { return Q[r + k * b]; }, lw, st);
  } else {
    const float *B = w.B + blockIdx.z * w.b_stride;
    gemm_block<kFactorTM, 16, true, true, false>(dj, g.r_max, s, m0, n0, [&](int64_t r, int64_t k) { return B[k + r * s]; }, lw, st);
  }
}

// ---------------------------------------------------------------- orthonormal basis
// Classical Gram-Schmidt with one reorthogonalisation, column by column, in
// place on Y (d_i x s). A column whose remainder after both passes is below
// 1e-5 of its own norm adds no direction the others do not hold to within
// fp32 rounding (there the second pass cannot restore orthogonality): it
// becomes zero, and its eigenvalue in the core is zero.
__global__ void __launch_bounds__(kOrthThreads) orth_kernel(Geo g, int64_t t0, Scratch w) {
  const int64_t t = t0 + blockIdx.x;
  const int64_t i = t / g.nJ, j = t % g.nJ;
  if (is_dense_tile(g, i, j)) return;
  const int64_t di = tile_dim(g.m, g.b, i);
  float *Q = w.Q + blockIdx.x * w.q_stride;
  const int64_t b = g.b;
  extern __shared__ float sm[];
  float *y = sm;                       // the current column (d_i <= b)
  float *coef = sm + b;                // kMaxSketch projections
  __shared__ float red[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = static_cast<int>(blockDim.x >> 5);
  auto sum_sq = [&]() {                // sum of y^2 over the block (every thread gets it)
    float a = 0.f;
    for (int64_t r = threadIdx.x; r < di; r += blockDim.x) a = fmaf(y[r], y[r], a);
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) red[warp] = a;
    __syncthreads();
    float tot = 0.f;
    for (int k = 0; k < nwarps; ++k) tot += red[k];
    __syncthreads();                   // red is reused by the next call
    return tot;
  };
  for (int c = 0; c < g.s; ++c) {
    for (int64_t r = threadIdx.x; r < di; r += blockDim.x) y[r] = Q[r + c * b];
    __syncthreads();
    const float orig2 = sum_sq();
    for (int pass = 0; pass < 2; ++pass) {
      // four independent partial sums per lane keep several loads of Q in flight
      for (int k = warp; k < c; k += nwarps) {
        const float *qk = Q + k * b;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        int64_t r = lane;
        for (; r + 96 < di; r += 128) {
          a0 = fmaf(qk[r], y[r], a0);
          a1 = fmaf(qk[r + 32], y[r + 32], a1);
          a2 = fmaf(qk[r + 64], y[r + 64], a2);
          a3 = fmaf(qk[r + 96], y[r + 96], a3);
        }
        for (; r < di; r += 32) a0 = fmaf(qk[r], y[r], a0);
        float a = (a0 + a1) + (a2 + a3);
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) coef[k] = a;
      }
      __syncthreads();
      for (int64_t r = threadIdx.x; r < di; r += blockDim.x) {
        float v0 = y[r], v1 = 0.f, v2 = 0.f, v3 = 0.f;
        int k = 0;
        for (; k + 3 < c; k += 4) {
          v0 = fmaf(-coef[k], Q[r + k * b], v0);
          v1 = fmaf(-coef[k + 1], Q[r + (k + 1) * b], v1);
          v2 = fmaf(-coef[k + 2], Q[r + (k + 2) * b], v2);
          v3 = fmaf(-coef[k + 3], Q[r + (k + 3) * b], v3);
        }
        for (; k < c; ++k) v0 = fmaf(-coef[k], Q[r + k * b], v0);
        y[r] = (v0 + v1) + (v2 + v3);
      }
      __syncthreads();
    }
    const float nrm2 = sum_sq();
    const float inv = nrm2 > 1e-10f * orig2 && nrm2 > 1e-36f ? rsqrtf(nrm2) : 0.f;
    for (int64_t r = threadIdx.x; r < di; r += blockDim.x) Q[r + c * b] = y[r] * inv;
    __syncthreads();
  }
}

// ---------------------------------------------------------------- eigen-decomposition of the core
// Cyclic Jacobi on G (s x s, s even) in shared memory, rows padded to s + 1
// floats. Each sweep runs s - 1 rounds of s/2 disjoint pairs (round-robin
// tournament: position 0 fixed, the others rotate); a round computes every
// pair's rotation, applies all of them to the rows (J^T G), then to the
// columns (G J) and to the accumulated eigenvectors (W J).
// kS: the sketch width when it is known when compiling (the row pitch kS + 1
// and the loop bounds become constants), 0 for any other width.
template <int kS>
__global__ void __launch_bounds__(kBigThreads) eig_kernel(Geo g, int64_t t0, Scratch w, int32_t *ranks, float *errors) {
  const int64_t t = t0 + blockIdx.x;
  const int64_t i = t / g.nJ, j = t % g.nJ;
  if (is_dense_tile(g, i, j)) {
    if (threadIdx.x == 0) { ranks[t] = 0; errors[t] = 0.f; }
    return;
  }
  const int s = kS ? kS : g.s, ps = s + 1;
  extern __shared__ float sm[];
  float *G = sm;                      // s x ps
  float *W = G + s * ps;              // s x ps
  float *lam = W + s * ps;            // s
  int *order = reinterpret_cast<int *>(lam + s);        // s
  const float *Gg = w.G + blockIdx.x * w.g_stride;
  for (int e = threadIdx.x; e < s * s; e += blockDim.x) {
    const int r = e % s, c = e / s;
    G[r * ps + c] = Gg[r + c * s];
    W[r * ps + c] = r == c ? 1.f : 0.f;
  }
  __syncthreads();
  // the trace (invariant under the rotations) sets the absolute scale
  __shared__ float trace_s;
  if (threadIdx.x == 0) {
    float tr = 0.f;
    for (int k = 0; k < s; ++k) tr += fabsf(G[k * ps + k]);
    trace_s = tr;
  }
  __syncthreads();
  const float floor_o = 2e-7f * trace_s;
  __shared__ int rotated;
  __shared__ int rot_pq[kMaxSketch / 2];   // a round's pairs (p | q << 16) and rotations
  __shared__ float rot_c[kMaxSketch / 2], rot_s[kMaxSketch / 2];
  for (int sweep = 0; sweep < 30; ++sweep) {
    // threshold Jacobi: a pair is rotated only while its off-diagonal entry is
    // above 1e-6 sqrt(|G_pp G_qq|), above the rounding level of its larger
    // diagonal entry and above 2e-7 of the trace (fp32 rounding of the core;
    // below that no energy the rank rule resolves can move); the sweeps end
    // when one rotates nothing
    if (threadIdx.x == 0) rotated = 0;
    __syncthreads();
    // Thread mapping: one warp per pair, warp w working on pairs w, w + 32,
    // ... in turn, its lanes on consecutive columns of a row (row update) or
    // consecutive rows of a column (column update); with the row pitch s + 1
    // both touch 32 distinct banks. Thread k < s / 2 computes the rotation of
    // pair k from the entries as they stand at the start of the round and
    // leaves it in a shared table for the warp working on that pair.
    const int half = s / 2;
    const int lane = static_cast<int>(threadIdx.x) & 31, warp = static_cast<int>(threadIdx.x) >> 5;
    for (int round = 0; round < s - 1; ++round) {
      // the round's rotations, one pair per thread of the first warps, into a
      // table the block reads after the barrier (the other warps issue none of
      // this arithmetic)
      if (static_cast<int>(threadIdx.x) < half) {
        const int kq = static_cast<int>(threadIdx.x);
        // round-robin order: position 0 stays, the others shift by one a round
        auto pos = [&](int x) {
          if (x == 0) return 0;
          const int y = x - 1 + round;
          return 1 + (y >= s - 1 ? y - (s - 1) : y);
        };
        int p = pos(kq), q = pos(s - 1 - kq);
        if (p > q) { const int tmp = p; p = q; q = tmp; }
        float cr = 1.f, sr = 0.f;
        const float a = G[p * ps + p], d = G[q * ps + q], o = G[p * ps + q];
        const float ao = fabsf(o);
        if (ao > 1e-6f * sqrtf(fabsf(a)) * sqrtf(fabsf(d)) && ao > 1e-7f * fmaxf(fabsf(a), fabsf(d)) &&
            ao > floor_o && ao > 1e-35f) {
          rotated = 1;
          // symmetric 2 x 2 Schur decomposition: t = tan(theta) with the smaller angle
          // |o| is above 2e-7 of the trace, so |tau| <= 2.5e6 and both fast
          // divisions stay far from their range limit
          const float tau = __fdividef(d - a, 2.f * o);
          const float tt = __fdividef(tau >= 0.f ? 1.f : -1.f, fabsf(tau) + sqrtf(1.f + tau * tau));
          cr = rsqrtf(1.f + tt * tt);
          sr = tt * cr;
        }
        rot_pq[kq] = p | (q << 16);
        rot_c[kq] = cr;
        rot_s[kq] = sr;
      }
      // the table is complete, and every read of the entries it came from is done
      __syncthreads();
      int pv[kPairsPerWarp], qv[kPairsPerWarp];
      float cv[kPairsPerWarp], sn[kPairsPerWarp];
#pragma unroll
      for (int m = 0; m < kPairsPerWarp; ++m) {
        const int kq = warp + m * kWarps;
        pv[m] = 0; qv[m] = 0; cv[m] = 1.f; sn[m] = 0.f;
        if (kq < half) {
          const int pq = rot_pq[kq];
          pv[m] = pq & 0xffff;
          qv[m] = pq >> 16;
          cv[m] = rot_c[kq];
          sn[m] = rot_s[kq];
        }
      }
      constexpr int kPer = kMaxSketch / 32;   // columns (rows) per lane
#pragma unroll
      for (int m = 0; m < kPairsPerWarp; ++m) {   // rows p, q of G
        if (sn[m] == 0.f) continue;
        const float c = cv[m], sv = sn[m];
        float *gp = G + pv[m] * ps, *gq = G + qv[m] * ps;
        float x[kPer], y[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e) {       // every load before any store
          const int col = lane + 32 * e;
          x[e] = col < s ? gp[col] : 0.f;
          y[e] = col < s ? gq[col] : 0.f;
        }
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          const int col = lane + 32 * e;
          if (col < s) {
            gp[col] = c * x[e] - sv * y[e];
            gq[col] = sv * x[e] + c * y[e];
          }
        }
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < kPairsPerWarp; ++m) {   // columns p, q of G and W
        if (sn[m] == 0.f) continue;
        const float c = cv[m], sv = sn[m];
        const int p = pv[m], q = qv[m];
        float x[kPer], y[kPer], u[kPer], v[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          const int row = lane + 32 * e;
          const bool in = row < s;
          x[e] = in ? G[row * ps + p] : 0.f;
          y[e] = in ? G[row * ps + q] : 0.f;
          u[e] = in ? W[row * ps + p] : 0.f;
          v[e] = in ? W[row * ps + q] : 0.f;
        }
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          const int row = lane + 32 * e;
          if (row < s) {
            G[row * ps + p] = c * x[e] - sv * y[e];
            G[row * ps + q] = sv * x[e] + c * y[e];
            W[row * ps + p] = c * u[e] - sv * v[e];
            W[row * ps + q] = sv * u[e] + c * v[e];
          }
        }
      }
      __syncthreads();
    }
    const int any = rotated;
    __syncthreads();   // every thread has read the flag before it is reset
    if (!any) break;
  }
  // eigenvalues (clamped at zero: the core is a Gram matrix) and their order
  for (int k = threadIdx.x; k < s; k += blockDim.x) lam[k] = fmaxf(G[k * ps + k], 0.f);
  __syncthreads();
  for (int k = threadIdx.x; k < s; k += blockDim.x) {
    int pos = 0;
    for (int q = 0; q < s; ++q) pos += lam[q] > lam[k] || (lam[q] == lam[k] && q < k);
    order[pos] = k;
  }
  __syncthreads();
  __shared__ int rank_s;
  if (threadIdx.x == 0) {
    const int64_t di = tile_dim(g.m, g.b, i), dj = tile_dim(g.n, g.b, j);
    int64_t cap = g.r_max;
    if (di < cap) cap = di;
    if (dj < cap) cap = dj;
    if (s < cap) cap = s;
    const double total = w.norm2[blockIdx.x];
    const double bound = static_cast<double>(g.eps) * static_cast<double>(g.eps) * total;
    double kept = 0.0;
    int r = 0;
    double tail = total;
    if (total > 0.0) {
      while (r < cap && tail > bound) {
        kept += lam[order[r]];
        ++r;
        tail = total - kept;
      }
    }
    if (tail < 0.0) tail = 0.0;
    ranks[t] = r;
    errors[t] = total > 0.0 ? static_cast<float>(sqrt(tail / total)) : 0.f;
    rank_s = r;
  }
  __syncthreads();
  const int r = rank_s;
  float *Wo = w.W + blockIdx.x * w.g_stride;
  float *lo = w.lam + blockIdx.x * static_cast<int64_t>(kMaxSketch);
  for (int e = threadIdx.x; e < s * s; e += blockDim.x) {
    const int row = e % s, k = e / s;
    Wo[row + k * s] = k < r ? W[row * ps + order[k]] : 0.f;
  }
  for (int k = threadIdx.x; k < s; k += blockDim.x) lo[k] = lam[order[k]];
}

// ---------------------------------------------------------------- dense tiles
__global__ void dense_copy_kernel(const float *C, int64_t ldc, Geo g, float *D) {
  const int64_t t = blockIdx.y;   // diagonal tile t
  const int64_t d = tile_dim(g.m, g.b, t);
  const float *T = C + t * g.b + t * g.b * ldc;
  float *o = D + t * g.b * g.b;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < d * d;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = e % d, c = e / d;
    o[r + c * g.b] = T[r + c * ldc];
  }
}

// ---------------------------------------------------------------- packing
struct CopyJob {
  const float *src;
  float *dst;
  int64_t rows, cols, src_ld, dst_ld;
};

__global__ void copy_jobs_kernel(const CopyJob *jobs, int njobs) {
  for (int jb = blockIdx.y; jb < njobs; jb += gridDim.y) {
    const CopyJob J = jobs[jb];
    const int64_t n = J.rows * J.cols;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const int64_t r = e % J.rows, c = e / J.rows;
      J.dst[r + c * J.dst_ld] = J.src[r + c * J.src_ld];
    }
  }
}

size_t eig_smem(int s) {
  const int ps = s + 1;
  return static_cast<size_t>(2 * s * ps + 2 * s) * 4;
}

}  // namespace tlr_cmp

using namespace tlr_cmp;

extern "C" {

tlr_status_t tlr_compress_workspace_bytes(int64_t b, int32_t s, int64_t tiles, size_t *bytes) {
  if (!bytes || b <= 0 || s <= 0 || tiles < 0) return TLR_STATUS_INVALID_ARG;
  const int64_t per = (2 * b * s + 2 * static_cast<int64_t>(s) * s + kMaxSketch) * 4 + 8;
  *bytes = static_cast<size_t>(per * std::max<int64_t>(tiles, 1) + 1024);
  return TLR_STATUS_OK;
}

tlr_status_t tlr_compress(tlr_handle_t h, const float *C, int64_t ldc, int64_t m, int64_t n, int64_t b,
                          int32_t dense_diagonal, float eps, int32_t r_max, const float *omega, int32_t s,
                          float *U, float *V, float *D, int32_t *ranks, float *errors, void *workspace,
                          size_t workspace_bytes) {
  if (!h) return TLR_STATUS_INVALID_ARG;
  if (m < 0 || n < 0 || b <= 0 || b > (1 << 20) || ldc < std::max<int64_t>(m, 1)) return TLR_STATUS_INVALID_ARG;
  if (s < 2 || s > kMaxSketch || (s & 1) || r_max < 0 || r_max > s) return TLR_STATUS_INVALID_ARG;
  if (!(eps >= 0.f) || !(eps < 1e30f)) return TLR_STATUS_INVALID_ARG;
  if (dense_diagonal && m != n) return TLR_STATUS_INVALID_ARG;
  if (m == 0 || n == 0) return TLR_STATUS_OK;
  if (!tlr::handle_on_current_device(h)) return TLR_STATUS_INVALID_ARG;
  const int64_t nI = (m + b - 1) / b, nJ = (n + b - 1) / b;
  if (nI * nJ > (int64_t(1) << 31)) return TLR_STATUS_INVALID_ARG;
  const bool need_f = r_max > 0 && !(dense_diagonal && nI == 1);
  if (!C || !omega || !ranks || !errors || !workspace || (need_f && (!U || !V)) || (dense_diagonal && !D))
    return TLR_STATUS_INVALID_ARG;
  const void *need[5] = {C, omega, ranks, errors, workspace};
  for (const void *p : need)
    if (!tlr::is_device_pointer(p)) return TLR_STATUS_INVALID_ARG;
  if ((need_f && (!tlr::is_device_pointer(U) || !tlr::is_device_pointer(V))) ||
      (dense_diagonal && !tlr::is_device_pointer(D)))
    return TLR_STATUS_INVALID_ARG;
  size_t per1 = 0;
  tlr_compress_workspace_bytes(b, s, 1, &per1);
  const int64_t per = static_cast<int64_t>(per1) - 1024;
  const int64_t ntiles = nI * nJ;
  const int64_t batch = std::min<int64_t>(ntiles, (static_cast<int64_t>(workspace_bytes) - 1024) / per);
  if (batch < 1) return TLR_STATUS_WORKSPACE_TOO_SMALL;
  cudaStream_t st = tlr::handle_stream(h);

  Geo g;
  g.m = m; g.n = n; g.b = b;
  g.nI = static_cast<int32_t>(nI); g.nJ = static_cast<int32_t>(nJ);
  g.dense_diag = dense_diagonal ? 1 : 0;
  g.s = s; g.r_max = r_max; g.eps = eps;

  // scratch of one batch, 256-byte aligned pieces
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255));
  Scratch w;
  w.q_stride = b * s;
  w.b_stride = static_cast<int64_t>(s) * b;
  w.g_stride = static_cast<int64_t>(s) * s;
  w.Q = reinterpret_cast<float *>(base);
  w.B = w.Q + batch * w.q_stride;
  w.G = w.B + batch * w.b_stride;
  w.W = w.G + batch * w.g_stride;
  w.lam = w.W + batch * w.g_stride;
  w.norm2 = reinterpret_cast<double *>(
      (reinterpret_cast<uintptr_t>(w.lam + batch * kMaxSketch) + 7) & ~uintptr_t(7));
  if (reinterpret_cast<uint8_t *>(w.norm2 + batch) > reinterpret_cast<uint8_t *>(workspace) + workspace_bytes)
    return TLR_STATUS_WORKSPACE_TOO_SMALL;

  const size_t esm = eig_smem(s);
  if (cudaFuncSetAttribute(eig_kernel<kMaxSketch>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(esm)) != cudaSuccess ||
      cudaFuncSetAttribute(eig_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(esm)) !=
          cudaSuccess)
    return TLR_STATUS_CUDA_ERROR;
  const size_t osm = static_cast<size_t>(b + kMaxSketch) * 4;
  if (osm > 227 * 1024) return TLR_STATUS_UNSUPPORTED;
  if (osm > 48 * 1024 &&
      cudaFuncSetAttribute(orth_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(osm)) !=
          cudaSuccess)
    return TLR_STATUS_CUDA_ERROR;

  // GEMM grids: blocks of (kernel's rows) x kTN columns
  auto blocks = [](int64_t n, int64_t per) { return static_cast<unsigned>((n + per - 1) / per); };
  const unsigned bN = blocks(b, kTN), sN = blocks(s, kTN), rN = blocks(std::max(r_max, 1), kTN);
  for (int64_t t0 = 0; t0 < ntiles; t0 += batch) {
    const unsigned nb = static_cast<unsigned>(std::min<int64_t>(batch, ntiles - t0));
    norm_kernel<<<nb, kBigThreads, 0, st>>>(C, ldc, g, t0, w);
    if (s > 64) sketch_kernel<128><<<dim3(blocks(b, kSketchTM), blocks(s, 128), nb), kThreads, 0, st>>>(C, ldc, omega, g, t0, w);
    else sketch_kernel<64><<<dim3(blocks(b, kSketchTM), sN, nb), kThreads, 0, st>>>(C, ldc, omega, g, t0, w);
    orth_kernel<<<nb, kOrthThreads, osm, st>>>(g, t0, w);
    project_kernel<<<dim3(blocks(s, kProjTM), bN, nb), kThreads, 0, st>>>(C, ldc, g, t0, w);
    core_kernel<<<dim3(blocks(s, kCoreTM), sN, nb), kThreads, 0, st>>>(g, t0, w);
    if (s == kMaxSketch) eig_kernel<kMaxSketch><<<nb, kBigThreads, esm, st>>>(g, t0, w, ranks, errors);
    else eig_kernel<0><<<nb, kBigThreads, esm, st>>>(g, t0, w, ranks, errors);
    if (r_max > 0) {
      factor_kernel<<<dim3(blocks(b, kFactorTM), rN, nb), kThreads, 0, st>>>(g, t0, w, U, V, 0);
      factor_kernel<<<dim3(blocks(b, kFactorTM), rN, nb), kThreads, 0, st>>>(g, t0, w, U, V, 1);
    }
    if (cudaGetLastError() != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  }
  if (dense_diagonal) {
    dense_copy_kernel<<<dim3(64, static_cast<unsigned>(nI)), kThreads, 0, st>>>(C, ldc, g, D);
    if (cudaGetLastError() != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  }
  return TLR_STATUS_OK;
}

tlr_status_t tlr_pack(tlr_handle_t h, int64_t n, int64_t b, int32_t r_max, const int32_t *ranks, const float *U_pad,
                      const float *V_pad, const float *D_pad, float *U, float *V, float *D, float *bu_U, float *bu_V,
                      float *bv_U, float *bv_V, float *gamma) {
  if (!h || !ranks || n <= 0 || b <= 0 || r_max < 0) return TLR_STATUS_INVALID_ARG;
  if (!tlr::handle_on_current_device(h)) return TLR_STATUS_INVALID_ARG;
  const int64_t mf = n / b, rem = n % b, nt = (n + b - 1) / b;
  bool lowrank = false, boundary_col = false, boundary_row = false;
  for (int64_t t = 0; t < nt * nt; ++t) {
    const int64_t i = t / nt, k = t % nt;
    if (ranks[t] < 0 || ranks[t] > r_max || (i == k && ranks[t] != 0)) return TLR_STATUS_INVALID_ARG;
    if (ranks[t] > 0) {
      lowrank = true;
      if (rem > 0 && k == mf) boundary_col = true;
      if (rem > 0 && i == mf) boundary_row = true;
    }
  }
  // every buffer a copy reads or writes must be there before any address is formed
  if (lowrank && (!U_pad || !V_pad)) return TLR_STATUS_INVALID_ARG;
  if (mf > 0 && (!D_pad || !D)) return TLR_STATUS_INVALID_ARG;
  if (rem > 0 && (!D_pad || !gamma)) return TLR_STATUS_INVALID_ARG;
  if (boundary_col && (!bu_U || !bu_V)) return TLR_STATUS_INVALID_ARG;
  if (boundary_row && (!bv_U || !bv_V)) return TLR_STATUS_INVALID_ARG;
  bool interior = false;
  for (int64_t i = 0; i < mf; ++i)
    for (int64_t k = 0; k < mf; ++k) interior = interior || ranks[i * nt + k] > 0;
  if (interior && (!U || !V)) return TLR_STATUS_INVALID_ARG;
  std::vector<CopyJob> jobs;
  auto add = [&](const float *src, float *dst, int64_t rows, int64_t cols, int64_t sld, int64_t dld) {
    if (rows > 0 && cols > 0) jobs.push_back(CopyJob{src, dst, rows, cols, sld, dld});
  };
  auto rk = [&](int64_t i, int64_t k) { return static_cast<int64_t>(ranks[i * nt + k]); };
  auto padU = [&](int64_t i, int64_t k) { return U_pad + (i * nt + k) * b * r_max; };
  auto padV = [&](int64_t i, int64_t k) { return V_pad + (i * nt + k) * b * r_max; };
  // interior: U by tile row, V by tile column
  int64_t off = 0;
  for (int64_t i = 0; i < mf; ++i)
    for (int64_t k = 0; k < mf; ++k)
      if (i != k && rk(i, k) > 0) { add(padU(i, k), U + off, b, rk(i, k), b, b); off += b * rk(i, k); }
  off = 0;
  for (int64_t k = 0; k < mf; ++k)
    for (int64_t i = 0; i < mf; ++i)
      if (i != k && rk(i, k) > 0) { add(padV(i, k), V + off, b, rk(i, k), b, b); off += b * rk(i, k); }
  for (int64_t t = 0; t < mf; ++t) add(D_pad + t * b * b, D + t * b * b, b, b, b, b);
  if (rem > 0) {
    int64_t ou = 0, ov = 0;
    for (int64_t i = 0; i < mf; ++i) {   // boundary column: tiles (i, mf)
      const int64_t r = rk(i, mf);
      if (r == 0) continue;
      add(padU(i, mf), bu_U + ou, b, r, b, b);
      add(padV(i, mf), bu_V + ov, rem, r, b, rem);
      ou += b * r; ov += rem * r;
    }
    ou = 0; ov = 0;
    for (int64_t j = 0; j < mf; ++j) {   // boundary row: tiles (mf, j)
      const int64_t r = rk(mf, j);
      if (r == 0) continue;
      add(padU(mf, j), bv_U + ou, rem, r, b, rem);
      add(padV(mf, j), bv_V + ov, b, r, b, b);
      ou += rem * r; ov += b * r;
    }
    add(D_pad + mf * b * b, gamma, rem, rem, b, rem);
  }
  for (const CopyJob &J : jobs)
    if (!J.dst || !J.src || !tlr::is_device_pointer(J.dst) || !tlr::is_device_pointer(J.src))
      return TLR_STATUS_INVALID_ARG;
  if (jobs.empty()) return TLR_STATUS_OK;
  cudaStream_t st = tlr::handle_stream(h);
  CopyJob *dj = nullptr;
  const size_t bytes = jobs.size() * sizeof(CopyJob);
  if (cudaMallocAsync(reinterpret_cast<void **>(&dj), bytes, st) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  // from pageable memory: the call returns once the jobs are staged
  if (cudaMemcpyAsync(dj, jobs.data(), bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  copy_jobs_kernel<<<dim3(16, static_cast<unsigned>(std::min<size_t>(jobs.size(), 65535))), kThreads, 0, st>>>(
      dj, static_cast<int>(jobs.size()));
  const bool ok = cudaGetLastError() == cudaSuccess;
  cudaFreeAsync(dj, st);
  return ok ? TLR_STATUS_OK : TLR_STATUS_CUDA_ERROR;
}

}  // extern "C"
