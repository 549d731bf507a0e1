// sm_103a kernels of the Tile-Low-Rank GEMM.
//
// tlr_task_gemm: a persistent, warp-specialised tensor-core GEMM that walks a
// table of output tiles ("tasks"). Each task accumulates, in tensor memory, the
// products of a short list of K segments; segment operands arrive through TMA
// tensor maps with exact extents, so ragged ranks are zero-filled on the fly and
// no factor is padded in memory. All stages of the method run through it:
//   Stage 1  S_k = V_{:,k}^T W_{k,:}                (one task group per k)
//   Stage 2  T_i[k-block, j-block] = S_ikj Z_kj^T   (fused over i, rows scattered)
//   Stage 3  C[i, J] = alpha U_i T_i (+ dense-tile segment) + beta C[i, J]
// ("Tile-Low-Rank GEMM: Designing Storage Around the Contraction", sections
// "One product, three stages" and "Where fusion stops"; the dense-diagonal
// terms follow "TLR Matrix Multiplication", section "Regular TLR GEMM").
//
// Roles (352 threads, one CTA per SM; instantiated for single CTAs, M = 128, and
// for CTA pairs, cta_group::2 with M = 256 across the two SMs):
//   warp 0       TMA producer: shared-memory ring of 4 stages (48 KiB) on a
//                single CTA or 6 stages (32 KiB) per CTA of a pair, 128-byte swizzle
//   warp 1       tcgen05.mma issuer (N = BN <= 256, fp32 accumulators in TMEM,
//                two accumulators so the epilogue of tile t overlaps tile t+1)
//   warp 2       descriptors: claims tickets, stages each task's segments, output
//                descriptor and per-row destinations in a shared-memory ring,
//                kRing tasks ahead
//   warps 3..10  epilogue, kEpiGroups groups of four warps (one per TMEM lane
//                quarter): tcgen05.ld, alpha/beta, stores staged through shared
//                memory (bulk tensor stores of C when beta == 0, 16-byte stores
//                of row-major 16-bit workspaces); group g takes the 64-column
//                blocks g, g + kEpiGroups, ... of the tile
// Every mbarrier wait is bounded (globaltimer); on timeout the CTA raises a flag
// in the device error word, drains its own copies and MMAs, frees TMEM, exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tlr_tables.h"

namespace tlr {

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on one phase of an mbarrier. Returns false when the limit ran
// out (the error word and the CTA's abort flag are then set) or when another
// role of this CTA already gave up.
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          const Params &p, uint32_t where, bool cluster_scope = false) {
  auto try_once = [&]() { return cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (try_once()) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (try_once()) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > p.wait_limit_ns) {
        *abort_flag = 1;
        atomicOr(p.err, 1u | (where << 4));
        return false;
      }
    }
  }
}

// Wait used while tearing down after an abort: ignores the abort flag.
__device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(unsigned int *p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait for a dependency counter (written by other CTAs of this launch).
__device__ __noinline__ bool wait_counter(const unsigned int *c, unsigned int target, volatile int *abort_flag,
                                          const Params &p) {
  if (ld_acquire(c) >= target) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ld_acquire(c) >= target) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > p.wait_limit_ns) {
        *abort_flag = 1;
        atomicOr(p.err, 1u | (9u << 4));
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Pair mode (cta_group::2): copies issued by either CTA of the pair complete on
// the leader CTA's mbarrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *tmap, int32_t x, int32_t y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// Pair mode with cluster multicast: the box lands at the same offset in every
// CTA of `mask`, and each destination's bytes complete on the mbarrier at the
// offset of `bar_cluster` in the leader CTA of that destination's pair.
__device__ __forceinline__ void tma_load_2d_pair_mc(uint32_t dst, const void *tmap, int32_t x, int32_t y,
                                                    uint32_t bar_cluster, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar_cluster), "h"(mask)
      : "memory");
}

// L2 policy for data written once and not read again in the launch (C): its
// lines are the first candidates for eviction, ahead of operands still in use.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void st_global_evict_first(void *ptr, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// Bulk tensor store of a shared-memory box (one thread), tracked per thread in bulk groups.
__device__ __forceinline__ void tma_store_2d(const void *tmap, uint32_t src, int32_t x, int32_t y, uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(src), "r"(x), "r"(y), "l"(pol)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Shared-memory source of every committed bulk store has been read.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every committed bulk store is complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Generic-proxy writes to shared memory become visible to bulk copies.
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of `addr` (a shared::cta address) in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family layout:
// start >> 4 in bits 0-13, leading byte offset >> 4 in 16-29, stride byte
// offset >> 4 in 32-45, version 1 in 46-47, swizzle mode 2 in 61-63).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor for kind::f16 (fp16 or bf16 inputs, both operands the
// same type) / kind::tf32, fp32 D.
__device__ __forceinline__ uint32_t idesc(bool tf32, bool f16, bool a_mn, bool b_mn, uint32_t n, uint32_t m = kBM) {
  const uint32_t fmt = tf32 ? 2u : (f16 ? 0u : 1u);   // tf32 / f16 / bf16
  uint32_t d = 0;
  d |= 1u << 4;                                   // D format: f32
  d |= fmt << 7;                                  // A format
  d |= fmt << 10;                                 // B format
  d |= (a_mn ? 1u : 0u) << 15;                    // A major: 0 K, 1 MN
  d |= (b_mn ? 1u : 0u) << 16;                    // B major
  d |= (n >> 3) << 17;                            // N / 8
  d |= (m >> 4) << 24;                            // M / 16
  return d;
}

template <bool kTF32>
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                    uint32_t accumulate) {
  if constexpr (kTF32) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
  }
}

template <bool kTF32>
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                         uint32_t accumulate) {
  if constexpr (kTF32) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
  }
}

// Commit for a pair: the mbarrier at the same offset in every CTA of `mask`
// (both CTAs of the pair by default) gets one arrival.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask = 0x3) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void mma_commit_pair_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 64 consecutive fp32 columns of this warp's 32 TMEM lanes. The wait is part of
// the same statement, so no use of the registers can be scheduled before it.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]),
        "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
        "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]),
        "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// One value as a 16-bit float (fp16 or bf16, round to nearest even), as raw bits.
__device__ __forceinline__ uint16_t to16(float x, bool f16) {
  return f16 ? __half_as_ushort(__float2half_rn(x)) : __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
// Two values as a packed pair of 16-bit floats (low half: a), one paired
// conversion instruction either way.
__device__ __forceinline__ uint32_t pack16x2(float a, float b, bool f16) {
  if (f16) {
    const __half2 h2 = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h2);
  }
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h2);
}

__device__ __forceinline__ float round_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// ------------------------------------------------------------------ the GEMM
// Stores one 32-column chunk of an output tile. Lane l of the warp holds the
// 32 accumulator values of tile row 32q + l (columns c0 .. c0 + nc - 1 of the
// output); `drow` is that row's destination (valid: the row is stored) and `stg`
// is the warp's 2 KiB staging area in shared memory.
// kRowIdx: rowd holds this lane's output rows for row-major 16-bit outputs
// (resolved once per task); otherwise they are shuffled out per chunk.
// kLoadC: with beta != 0, each half's C is loaded before any of it is stored
// (more registers; the fp32-input kernels, whose products carry beta != 0).
template <bool kRowIdx, bool kLoadC>
__device__ __forceinline__ void store_chunk(float (&v)[32], int nc, int64_t c0, int64_t drow, bool valid,
                                            const Params &p, const Out &o, int lane, uint8_t *stg,
                                            const int32_t (&rowd)[4], bool &bulk_live) {
  if (o.kind == kOutC) {
    // fp32 C through shared memory in two 16-column halves. The warp's block is
    // 32 rows x 16 columns of column-major C (tile rows are rows of C), or 16
    // rows x 32 columns (transposed tile: tile row r is column drow(r) of C,
    // tile columns are its rows). With beta == 0 and a whole block inside the
    // task, one bulk tensor store writes it; otherwise every store instruction
    // writes 16 contiguous bytes per lane (4 columns x 128 bytes, or 8 columns
    // x 64 bytes), and C is read the same way when beta != 0.
    float *C = p.C;
    const int64_t ld = p.ldc;
    const int64_t d0 = __shfl_sync(0xffffffffu, drow, 0);
    const bool contiguous = __all_sync(0xffffffffu, valid && drow == d0 + lane);
    const bool rows_ok = contiguous && (d0 & 3) == 0;
    const bool fast = o.trans ? (nc & 3) == 0 : rows_ok;
    // bulk stores need the box's first row (the map's inner coordinate) on a 16-byte boundary
    const bool bulk = p.cmap_ok && p.beta == 0.f && contiguous && ((o.trans ? c0 : d0) & 3) == 0;
    if (fast) {
      float *sf = reinterpret_cast<float *>(stg);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int nch = nc - 16 * h < 16 ? nc - 16 * h : 16;   // columns of this half
        if (nch <= 0) break;
        if (bulk_live) {   // an earlier bulk store may still be reading the staging area
          if (lane == 0) bulk_wait_read();
          __syncwarp();
          bulk_live = false;
        }
        // with beta != 0 this half's C is loaded before any of it is stored, all
        // four loads in flight at once (a load after a store to C could not be
        // issued early), once the values are parked and their registers free
        float4 cv[4];
        if (!o.trans) {
#pragma unroll
          for (int j = 0; j < 16; ++j) sf[j * 32 + lane] = p.alpha * v[16 * h + j];   // [column][row]
          if (kLoadC && p.beta != 0.f) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const int j = 4 * s + (lane >> 3), r4 = 4 * (lane & 7);
              if (j < nch) cv[s] = *reinterpret_cast<const float4 *>(C + d0 + r4 + (c0 + 16 * h + j) * ld);
            }
          }
          if (bulk && nch == 16) {
            fence_async_shared();
            __syncwarp();
            if (lane == 0) tma_store_2d(&p.cmap[0], smem_u32(sf), static_cast<int32_t>(d0),
                                        static_cast<int32_t>(c0 + 16 * h), policy_evict_first());
            bulk_live = true;
            continue;
          }
          __syncwarp();
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const int j = 4 * s + (lane >> 3), r4 = 4 * (lane & 7);
            if (j < nch) {
              float4 x = *reinterpret_cast<const float4 *>(sf + j * 32 + r4);
              float4 *dst = reinterpret_cast<float4 *>(C + d0 + r4 + (c0 + 16 * h + j) * ld);
              if (p.beta != 0.f) {
                const float4 c = kLoadC ? cv[s] : *dst;
                x.x = fmaf(p.beta, c.x, x.x); x.y = fmaf(p.beta, c.y, x.y);
                x.z = fmaf(p.beta, c.z, x.z); x.w = fmaf(p.beta, c.w, x.w);
              }
              *dst = x;
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<float4 *>(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
                make_float4(p.alpha * v[16 * h + 4 * c], p.alpha * v[16 * h + 4 * c + 1],
                            p.alpha * v[16 * h + 4 * c + 2], p.alpha * v[16 * h + 4 * c + 3]);
          int64_t dd[4];
          if constexpr (kLoadC) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const int r = 8 * s + (lane >> 2), c = lane & 3;
              dd[s] = __shfl_sync(0xffffffffu, valid ? drow : int64_t(-1), r);
              if (p.beta != 0.f && dd[s] >= 0 && 4 * c < nch)
                cv[s] = *reinterpret_cast<const float4 *>(C + (c0 + 16 * h + 4 * c) + dd[s] * ld);
            }
          }
          if (bulk && nch == 16) {   // the XOR layout above is the map's 64-byte swizzle
            fence_async_shared();
            __syncwarp();
            if (lane == 0) tma_store_2d(&p.cmap[1], smem_u32(stg), static_cast<int32_t>(c0 + 16 * h),
                                        static_cast<int32_t>(d0), policy_evict_first());
            bulk_live = true;
            continue;
          }
          __syncwarp();
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const int r = 8 * s + (lane >> 2), c = lane & 3;
            float4 x = *reinterpret_cast<const float4 *>(stg + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
            int64_t d;
            if constexpr (kLoadC) d = dd[s];
            else d = __shfl_sync(0xffffffffu, valid ? drow : int64_t(-1), r);
            if (d >= 0 && 4 * c < nch) {
              float4 *dst = reinterpret_cast<float4 *>(C + (c0 + 16 * h + 4 * c) + d * ld);
              if (p.beta != 0.f) {
                const float4 cw = kLoadC ? cv[s] : *dst;
                x.x = fmaf(p.beta, cw.x, x.x); x.y = fmaf(p.beta, cw.y, x.y);
                x.z = fmaf(p.beta, cw.z, x.z); x.w = fmaf(p.beta, cw.w, x.w);
              }
              *dst = x;
            }
          }
        }
        __syncwarp();   // the staging area is reused by the next half
      }
      return;
    }
  }
  if (o.kind == kOutC && o.trans) {
    // Ragged transposed tile: transpose the warp's 32 x 32 block across lanes
    // (XOR butterfly) so that lane i holds tile column c0 + i for the warp's 32
    // rows; every store then writes consecutive floats of one column of C.
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
      const bool upper = (lane & sh) != 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j & sh) continue;
        const float send = upper ? v[j] : v[j | sh];
        const float recv = __shfl_xor_sync(0xffffffffu, send, sh);
        if (upper) v[j] = recv;
        else v[j | sh] = recv;
      }
    }
    float *C = p.C;
    const int64_t ld = p.ldc;
    const bool cok = lane < nc;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int64_t dj = __shfl_sync(0xffffffffu, valid ? drow : int64_t(-1), j);
      if (cok && dj >= 0) {
        const int64_t off = (c0 + lane) + dj * ld;
        float val = p.alpha * v[j];
        if (p.beta != 0.f) val = fmaf(p.beta, C[off], val);
        C[off] = val;
      }
    }
    return;
  }
  const bool half16 = o.kind == kOutBF16 || o.kind == kOutF16;   // 16-bit workspace output
  if (half16 && o.trans && nc == 32) {
    // Row-major 16-bit output through shared memory: each lane parks its row's
    // 64 bytes (16-byte chunks XOR-swizzled by row pair, so neither the writes
    // nor the reads conflict on banks); then each store instruction writes
    // 8 rows x 64 contiguous bytes instead of 32 rows x 16 bytes.
    if (bulk_live) {   // an earlier bulk store may still be reading the staging area
      if (lane == 0) bulk_wait_read();
      __syncwarp();
      bulk_live = false;
    }
    uint32_t pk[16];
    if (o.kind == kOutF16) {   // one conversion per branch, decided once per chunk
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] = pack16x2(v[2 * i], v[2 * i + 1], true);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] = pack16x2(v[2 * i], v[2 * i + 1], false);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4 *>(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
          make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    __syncwarp();
    const uint64_t pol = policy_evict_first();
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int r = 8 * s + (lane >> 2), c = lane & 3;
      const uint4 val = *reinterpret_cast<const uint4 *>(stg + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
      // rowd[s]: output row of row 8s + lane/4 of this warp's block (-1: not
      // stored), resolved once per task. A rectangle's T is larger than L2 and
      // is read back only by its final products, after every Stage-2 tile of
      // the rectangle: its lines go first, ahead of the operands being reused now.
      int64_t d;
      if constexpr (kRowIdx) d = rowd[s];
      else d = __shfl_sync(0xffffffffu, valid ? drow : int64_t(-1), r);
      if (d >= 0) st_global_evict_first(static_cast<uint16_t *>(o.ptr) + d * o.ld + c0 + 8 * c, val, pol);
    }
    __syncwarp();   // the staging area is reused by the next chunk
    return;
  }
  if (!valid) return;
  if (o.kind == kOutC) {
    float *C = p.C;
    const int64_t ld = p.ldc;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < nc) {
        const int64_t off = drow + (c0 + i) * ld;
        float val = p.alpha * v[i];
        if (p.beta != 0.f) val = fmaf(p.beta, C[off], val);
        C[off] = val;
      }
    }
  } else if (half16) {
    uint16_t *W = static_cast<uint16_t *>(o.ptr);
    uint16_t h[32];
    if (o.kind == kOutF16) {
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = to16(v[i], true);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = to16(v[i], false);
    }
    if (o.trans) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nc) W[drow * o.ld + c0 + i] = h[i];
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nc) W[drow + (c0 + i) * o.ld] = h[i];
    }
  } else {
    float *W = static_cast<float *>(o.ptr);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nc) W[o.trans ? (c0 + i) + drow * o.ld : drow + (c0 + i) * o.ld] = round_tf32(v[i]);
  }
}

// One staged task in shared memory (written by the descriptor warp).
struct Slot {
  Task task;                 // 48 B
  Out out;                   // 32 B
  int32_t pad_[4];
  Seg segs[kMaxSegs];        // at 96
  int64_t pad2_[4];
  int64_t rowdst[kBM];       // at 384: output row of each tile row, -1 when the row is not stored
};
static_assert(sizeof(Slot) <= kSlotBytes, "slot size");

template <bool kTF32, int kPair>
__global__ void __launch_bounds__(kThreads, 1) tlr_task_gemm(const __grid_constant__ Params p) {
  static_assert(kPair == 1 || kPair == 2 || kPair == 4, "one CTA, a CTA pair, or two pairs per cluster");
  // kPair == 2: the tile is 256 rows; each CTA of the pair holds 128 rows of A and
  // half of the columns of B; the leader issues cta_group::2 MMAs into both TMEMs.
  // kPair == 4: a cluster of two such pairs working on tiles that share their B
  // operand (tickets 8g..8g+3 for the first pair, 8g+4..8g+7 for the second, slot
  // by slot with equal B segments): the first pair loads B once and multicasts it
  // into the second pair's shared memory, so the cluster reads 3/4 of the operand
  // bytes two separate pairs would.
  constexpr bool kCG2 = kPair >= 2;                       // cta_group::2 MMAs over a CTA pair
  constexpr bool kQuad = kPair == 4;
  constexpr int kPairCTAs = kCG2 ? 2 : 1;                 // CTAs per output tile
  constexpr int kSt = kCG2 ? 6 : kStages;                 // pipeline stages
  constexpr int kStB = kSmemA + kMaxBN / kPairCTAs * 128; // bytes per stage in this CTA
  static_assert(kSt * kStB == kStages * kStageBytes, "same shared-memory footprint");
  constexpr int kElt = kTF32 ? 4 : 2;
  constexpr int kCH = 128 / kElt;     // elements per 128-byte row: MN chunk and K block
  constexpr int kBK = kCH;
  constexpr int kUK = 32 / kElt;      // K of one MMA instruction (32 bytes)

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *base_ptr = smem_raw + (base - raw);
  Slot *ring = reinterpret_cast<Slot *>(base_ptr + kSt * kStB);
  const uint32_t bars = base + kSt * kStB + kRing * kSlotBytes;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kSt + s); };
  auto tfull_bar = [&](int a) { return bars + 8u * (2 * kSt + a); };
  auto tempty_bar = [&](int a) { return bars + 8u * (2 * kSt + kMaxAcc + a); };
  const uint32_t drain_bar = bars + 8u * (2 * kSt + 2 * kMaxAcc);
  auto sfull_bar = [&](int r) { return bars + 8u * (2 * kSt + 2 * kMaxAcc + 1 + r); };
  auto sempty_bar = [&](int r) { return bars + 8u * (2 * kSt + 2 * kMaxAcc + 1 + kRing + r); };
  const uint32_t sig_bar = bars + 8u * (2 * kSt + 2 * kMaxAcc + 1 + 2 * kRing);   // epilogue stores published
  static_assert(8 * (2 * kSt + 2 * kMaxAcc + 2 + 2 * kRing) + 16 <= 512, "barrier area");
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(base_ptr + kSt * kStB + kRing * kSlotBytes +
                                                       8 * (2 * kSt + 2 * kMaxAcc + 2 + 2 * kRing));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bn = p.bn;
  // TMEM holds kTmemCols fp32 columns: two accumulators of 256 columns, or four
  // of 128 for tiles at most 128 wide, so that the MMAs of up to three tiles
  // proceed while the epilogue drains the fourth
  const int nacc = bn <= kMaxBN / 2 ? 4 : 2;
  const uint32_t acc_cols = static_cast<uint32_t>(kTmemCols / nacc);
  const uint32_t crank = kCG2 ? cluster_rank() : 0u;      // rank in the cluster
  const uint32_t rank = crank & 1u;                        // rank in the pair; 0: leader of the pair
  const uint32_t lead_rank = crank & ~1u;                  // cluster rank of this pair's leader
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kQuad ? 2 : 1);   // quad: both pairs' MMAs release a stage
    }
    for (int a = 0; a < kMaxAcc; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4 * kEpiGroups * kPairCTAs);   // one arrival per epilogue warp of the pair
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(sfull_bar(r), 1);
      mbar_init(sempty_bar(r), 2 + 4 * kEpiGroups);   // producer, MMA issuer, every epilogue warp
    }
    mbar_init(drain_bar, 1);
    mbar_init(sig_bar, kEpiThreads);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    if constexpr (kCG2) {
      // one warp of each CTA of the pair allocates collectively
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_holder)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_holder)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kCG2) cluster_sync_all();   // the peers' barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const char *maps = reinterpret_cast<const char *>(p.maps);

  if (warp == 2) {
    // ---------------------------------------------------------------- descriptors
    // Claim tickets in batches of kBatch (one CTA: from a global counter; a pair:
    // batches pair, pair + npairs, ...; every pair is resident, so a dependency
    // on a lower ticket is always met), load the batch's task headers in parallel,
    // then per task: wait for its dependencies, load its segments, output
    // descriptor and row pieces in one parallel round, resolve the destination of
    // each tile row with shuffles and stage everything in ring slot n % kRing.
    // A slot whose task has nseg < 0 tells the consumers there is no more work.
    constexpr int kBatch = kTicketBatch;
    int n = 0;
    bool done = false;
    // One CTA claims kBatch tickets at a time from the launch's counter. CTA
    // pairs take their tickets in a fixed order: whole rounds of kBatch-ticket
    // batches, then the remainder one ticket per pair in turn, so the pairs
    // finish within about one task of each other (with batches throughout, the
    // last round left half the pairs idle for up to kBatch final-product tiles).
    const unsigned int ntasks = static_cast<unsigned int>(p.ntasks);
    for (uint32_t b = 0; !done; ++b) {
      unsigned int t0 = 0, cnt = kBatch;
      if (lane == 0) {
        if constexpr (kPair == 1) {
          t0 = atomicAdd(p.ticket, cnt);
        } else if constexpr (kQuad) {
          // whole groups of 2 kBatch tickets per cluster in turn; the planner pads
          // the launch to whole groups
          const unsigned int units = gridDim.x / 4, unit = blockIdx.x / 4;
          t0 = ((unit + b * units) * 2 + (crank >> 1)) * kBatch;
        } else {
          const unsigned int units = gridDim.x / 2, unit = blockIdx.x / 2;
          const unsigned int rounds = ntasks / (kBatch * units);
          if (b < rounds) {
            t0 = (unit + b * units) * kBatch;
          } else {
            t0 = rounds * kBatch * units + unit + (b - rounds) * units;
            cnt = 1;
          }
        }
      }
      t0 = __shfl_sync(0xffffffffu, t0, 0);
      cnt = __shfl_sync(0xffffffffu, cnt, 0);
      Task mine;
      if (lane < static_cast<int>(cnt) && t0 + lane < ntasks) mine = p.tasks[t0 + lane];
      for (int j = 0; j < static_cast<int>(cnt); ++j, ++n) {
        const int r = n % kRing;
        const uint32_t ph = (n / kRing) & 1;
        Slot &sl = ring[r];
        int ok = 1;
        if (lane == 0) ok = wait_bounded(sempty_bar(r), ph ^ 1u, abort_flag, p, 5) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) { done = true; break; }
        if (t0 + j >= static_cast<unsigned int>(p.ntasks)) {
          if (lane == 0) {
            sl.task.nseg = -1;
            mbar_arrive(sfull_bar(r));
          }
          done = true;
          break;
        }
        // broadcast task j's header from lane j
        Task task;
        {
          const int32_t *src = reinterpret_cast<const int32_t *>(&mine);
          int32_t *dst = reinterpret_cast<int32_t *>(&task);
#pragma unroll
          for (int w = 0; w < static_cast<int>(sizeof(Task) / 4); ++w) dst[w] = __shfl_sync(0xffffffffu, src[w], j);
        }
        // one parallel round of loads: output descriptor, segments, row pieces
        Out out;
        if (lane == 0) out = p.outs[task.out];
        Seg sg;
        if (lane < task.nseg) sg = p.segs[task.seg0 + lane];
        Piece pe;
        pe.src0 = 0; pe.len = 0; pe.dst0 = 0;
        const int np = task.npiece < 32 ? task.npiece : 32;
        if (lane < np) pe = p.pieces[task.piece0 + lane];
        if (lane == 0) {
          for (int d = 0; d < 2 && ok; ++d)
            if (task.dep[d] >= 0) ok = wait_counter(p.counters + task.dep[d], task.dep_target[d], abort_flag, p) ? 1 : 0;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) { done = true; break; }
        if (lane == 0) { sl.task = task; sl.out = out; }
        if (lane < task.nseg) sl.segs[lane] = sg;
        int64_t d[kBM / 32];
#pragma unroll
        for (int q4 = 0; q4 < kBM / 32; ++q4) {
          const int trow = static_cast<int>(rank) * kBM + q4 * 32 + lane;   // row of the (pair) tile
          d[q4] = trow < task.rows && task.npiece == 0 ? task.row0 + trow : -1;
        }
        if (task.npiece > 0) {
          for (int base_p = 0; base_p < task.npiece; base_p += 32) {
            if (base_p > 0) {   // more than 32 pieces: next round
              const int m = task.npiece - base_p < 32 ? task.npiece - base_p : 32;
              pe.src0 = 0; pe.len = 0; pe.dst0 = 0;
              if (lane < m) pe = p.pieces[task.piece0 + base_p + lane];
            }
            const int m = task.npiece - base_p < 32 ? task.npiece - base_p : 32;
            for (int q = 0; q < m; ++q) {
              const int32_t s0 = __shfl_sync(0xffffffffu, pe.src0, q);
              const int32_t ln = __shfl_sync(0xffffffffu, pe.len, q);
              const int64_t d0 = __shfl_sync(0xffffffffu, pe.dst0, q);
#pragma unroll
              for (int q4 = 0; q4 < kBM / 32; ++q4) {
                const int trow = static_cast<int>(rank) * kBM + q4 * 32 + lane;
                if (trow < task.rows && trow >= s0 && trow < s0 + ln) d[q4] = d0 + (trow - s0);
              }
            }
          }
        }
#pragma unroll
        for (int q4 = 0; q4 < kBM / 32; ++q4) sl.rowdst[q4 * 32 + lane] = d[q4];
        __syncwarp();
        if (lane == 0) mbar_arrive(sfull_bar(r));
      }
    }
  } else if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_phase_mask = 0;   // per stage: copy issued / its phase
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const int r = n % kRing;
        if (!wait_bounded(sfull_bar(r), (n / kRing) & 1, abort_flag, p, 6)) break;
        const Slot &sl = ring[r];
        const int nseg = sl.task.nseg;
        if (nseg < 0) break;
        // operands written earlier in this launch by other CTAs are read through TMA
        if (sl.task.dep[0] >= 0 || sl.task.dep[1] >= 0) fence_proxy_async_global();
        for (int s = 0; ok && s < nseg; ++s) {
          const Seg sg = sl.segs[s];
          const void *ma = maps + 128 * static_cast<size_t>(sg.a_map);
          const void *mb = maps + 128 * static_cast<size_t>(sg.b_map);
          const int nkb = (sg.k_len + kBK - 1) / kBK;
          // Box walk of each operand: MN-major boxes are kCH wide along MN (x) and
          // step K along y; K-major boxes are 64 rows along MN (y) and step K along x.
          const int32_t am0 = static_cast<int32_t>(rank) * kBM;   // this CTA's rows of A
          const int bnc = bn / kPairCTAs;                         // this CTA's columns of B
          const int32_t bn0 = static_cast<int32_t>(rank) * bnc;
          const bool amn = (sg.flags & kSegAMN) != 0, bmn = (sg.flags & kSegBMN) != 0;
          int32_t ax = amn ? sg.a_x + am0 : sg.a_x, ay = amn ? sg.a_y : sg.a_y + am0;
          int32_t bx = bmn ? sg.b_x + bn0 : sg.b_x, by = bmn ? sg.b_y : sg.b_y + bn0;
          const int32_t adx = amn ? kCH : 0, ady = amn ? 0 : 64, akx = amn ? 0 : kBK, aky = amn ? kBK : 0;
          const int32_t bdx = bmn ? kCH : 0, bdy = bmn ? 0 : 64, bkx = bmn ? 0 : kBK, bky = bmn ? kBK : 0;
          const int nba = amn ? kBM / kCH : kBM / 64, nbb = bmn ? bnc / kCH : bnc / 64;
          const uint32_t sta = amn ? kBK * 128 : 64 * 128, stb = sta;
          for (int kb = 0; kb < nkb; ++kb) {
            const uint32_t eb = empty_bar(stage);
            if (!mbar_try_wait(eb, phase ^ 1u) && !wait_bounded(eb, phase ^ 1u, abort_flag, p, 1)) { ok = false; break; }
            const uint32_t fb = full_bar(stage);
            // one CTA: its own barrier; a pair: both CTAs' copies complete on the leader's
            // barrier, which the leader arms with the bytes of both
            if (leader) mbar_expect_tx(fb, kPairCTAs * kSmemA + bn * 128);
            const uint32_t fb_tma = kCG2 ? map_to_rank(fb, lead_rank) : fb;
            const uint32_t sa = base + stage * kStB;
            const uint32_t sb = sa + kSmemA;
            for (int c = 0; c < nba; ++c) {
              if constexpr (kCG2) tma_load_2d_pair(sa + c * sta, ma, ax + c * adx, ay + c * ady, fb_tma);
              else tma_load_2d(sa + c * sta, ma, ax + c * adx, ay + c * ady, fb_tma);
            }
            if (!kQuad || crank < 2) {   // quad: the first pair's CTAs load B for both pairs
              for (int c = 0; c < nbb; ++c) {
                if constexpr (kQuad)
                  tma_load_2d_pair_mc(sb + c * stb, mb, bx + c * bdx, by + c * bdy, fb_tma,
                                      static_cast<uint16_t>((1u << crank) | (1u << (crank + 2))));
                else if constexpr (kCG2) tma_load_2d_pair(sb + c * stb, mb, bx + c * bdx, by + c * bdy, fb_tma);
                else tma_load_2d(sb + c * stb, mb, bx + c * bdx, by + c * bdy, fb_tma);
              }
            }
            ax += akx; ay += aky; bx += bkx; by += bky;
            issued_mask |= 1u << stage;
            issued_phase_mask = (issued_phase_mask & ~(1u << stage)) | (phase << stage);
            if (++stage == kSt) { stage = 0; phase ^= 1u; }
          }
        }
        mbar_arrive(sempty_bar(r));
      }
      // Every copy this thread issued must land before the CTA may exit (a pair's
      // copies complete on the leader's barriers; the peer leaves after the leader
      // at the final cluster barrier).
      if (leader)
        for (int s = 0; s < kSt; ++s)
          if (issued_mask & (1u << s)) wait_drain(full_bar(s), (issued_phase_mask >> s) & 1u, 200000000ull);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const int r = n % kRing;
        if (!wait_bounded(sfull_bar(r), (n / kRing) & 1, abort_flag, p, 7)) break;
        const Slot &sl = ring[r];
        const int nseg = sl.task.nseg;
        if (nseg < 0) break;
        if (kCG2 && !leader) {   // the peer's MMA warp only walks the ring
          mbar_arrive(sempty_bar(r));
          continue;
        }
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p, 2, kCG2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * acc_cols;
        uint32_t accumulate = 0;
        for (int s = 0; ok && s < nseg; ++s) {
          const Seg sg = sl.segs[s];
          const bool a_mn = sg.flags & kSegAMN, b_mn = sg.flags & kSegBMN;
          const uint32_t id = idesc(kTF32, p.f16 != 0, a_mn, b_mn, static_cast<uint32_t>(bn), kBM * kPairCTAs);
          const int nkb = (sg.k_len + kBK - 1) / kBK;
          // Descriptors of stage 0; a stage is kStB bytes further, an MMA step 32 bytes
          // (K-major: the next K slice of each 128-byte swizzled row) or kUK rows of
          // 128 bytes (MN-major: whole 8-row groups). The start address sits in the
          // low 14 bits (>> 4), so steps are plain additions.
          const uint64_t a0 = a_mn ? sdesc(base, kBK * 128, 1024) : sdesc(base, 16, 1024);
          const uint64_t b0 = b_mn ? sdesc(base + kSmemA, kBK * 128, 1024) : sdesc(base + kSmemA, 16, 1024);
          const uint64_t da = a_mn ? (kUK * 128) >> 4 : 32 >> 4, db = b_mn ? (kUK * 128) >> 4 : 32 >> 4;
          constexpr uint64_t dst = kStB >> 4;
          for (int kb = 0; kb < nkb; ++kb) {
            const uint32_t fb = full_bar(stage);
            if (!mbar_try_wait(fb, phase) && !wait_bounded(fb, phase, abort_flag, p, 3)) { ok = false; break; }
            tc_fence_after();
            const uint64_t ad = a0 + stage * dst, bd = b0 + stage * dst;
            const int kleft = sg.k_len - kb * kBK;
            if (kleft >= kBK) {
#pragma unroll
              for (int k = 0; k < kBK / kUK; ++k) {
                if constexpr (kCG2) mma_pair<kTF32>(d_tmem, ad + k * da, bd + k * db, id, accumulate);
                else mma<kTF32>(d_tmem, ad + k * da, bd + k * db, id, accumulate);
                accumulate = 1;
              }
            } else {
              const int nmma = (kleft + kUK - 1) / kUK;
              for (int k = 0; k < nmma; ++k) {
                if constexpr (kCG2) mma_pair<kTF32>(d_tmem, ad + k * da, bd + k * db, id, accumulate);
                else mma<kTF32>(d_tmem, ad + k * da, bd + k * db, id, accumulate);
                accumulate = 1;
              }
            }
            // frees the stage (in both CTAs of a pair, in all four of a quad) once these MMAs have read it
            if constexpr (kQuad) mma_commit_pair(empty_bar(stage), 0xF);
            else if constexpr (kCG2) mma_commit_pair(empty_bar(stage));
            else mma_commit(empty_bar(stage));
            if (++stage == kSt) { stage = 0; phase ^= 1u; }
          }
        }
        mbar_arrive(sempty_bar(r));
        if (!ok) break;
        if (accumulate) {
          if constexpr (kCG2) mma_commit_pair(tfull_bar(acc), static_cast<uint16_t>(0x3u << lead_rank));
          else mma_commit(tfull_bar(acc));
        } else {
          mbar_arrive(tfull_bar(acc));
          if constexpr (kCG2) mbar_arrive_remote(map_to_rank(tfull_bar(acc), lead_rank + 1));
        }
        if (++acc == nacc) { acc = 0; acc_phase ^= 1u; }
      }
      // All MMAs issued by this thread complete before TMEM is released.
      if (leader) {
        if constexpr (kCG2) mma_commit_pair_local(drain_bar);
        else mma_commit(drain_bar);
        wait_drain(drain_bar, 0, 200000000ull);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;               // TMEM lanes 32q..32q+31 belong to this warp
    const int row = q * 32 + lane;        // accumulator row held by this thread
    const int grp = (warp - 3) >> 2;      // epilogue group: its share of the 64-column chunks
    uint8_t *stg = base_ptr + kSt * kStB + kRing * kSlotBytes + 512 + (warp - 3) * kEpiStageBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    // Completion signals are per warp and batched: consecutive tasks that
    // signal the same counter add their counts and publish them with one fence.
    // A warp publishes what it holds before it would block (next task not yet
    // staged, accumulator not yet ready), when the counter changes, and every
    // kSignalBatch tasks, so a dependency on its tasks can always be met.
    bool bulk_live = false;               // this warp has bulk stores that may still read its staging area
    int32_t pend = -1;
    uint32_t pend_n = 0;
    bool pend_writes = false;
    auto flush = [&]() {
      if (pend < 0) return;
      if (pend_writes) {
        fence_proxy_async_global();   // publish this lane's stores to TMA readers
        __threadfence();
      }
      __syncwarp();
      if (lane == 0) red_release_add(p.counters + pend, pend_n);
      pend = -1;
      pend_n = 0;
      pend_writes = false;
    };
    auto ready = [&](uint32_t bar, uint32_t parity) {
      const uint32_t ok = lane == 0 ? (kCG2 ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) : 0u;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    for (int n = 0;; ++n) {
      const int r = n % kRing;
      if (!ready(sfull_bar(r), (n / kRing) & 1)) flush();
      if (!wait_bounded(sfull_bar(r), (n / kRing) & 1, abort_flag, p, 8)) break;
      const Slot &sl = ring[r];
      if (sl.task.nseg < 0) break;
      const int32_t signal = sl.task.signal;
      const bool signal_writes = sl.task.signal_writes != 0;
      const int64_t drow = sl.rowdst[row];
      const bool valid = drow >= 0;
      const int ncols = sl.task.cols;
      const bool has_acc = sl.task.nseg > 0;
      const int64_t col0 = sl.task.col0;
      const Out o = sl.out;
      __syncwarp();
      if (lane == 0) mbar_arrive(sempty_bar(r));
      if (!ready(tfull_bar(acc), acc_phase)) flush();
      if (!wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p, 4, kCG2)) break;
      tc_fence_after();
      if (pend != signal || pend_n >= kSignalBatch) flush();   // the earlier stores have had time to drain
      const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                              static_cast<uint32_t>(acc) * acc_cols;
      // row-major 16-bit outputs: the output rows of this lane's four 16-byte
      // pieces of every chunk (workspace rows fit in 32 bits)
      int32_t rowd[4] = {-1, -1, -1, -1};
      if (kPair == 1 && (o.kind == kOutBF16 || o.kind == kOutF16) && o.trans) {
        const int32_t dr = valid ? static_cast<int32_t>(drow) : -1;
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) rowd[s4] = __shfl_sync(0xffffffffu, dr, 8 * s4 + (lane >> 2));
      }
      for (int cc = 64 * grp; cc < ncols; cc += 64 * kEpiGroups) {
        float v64[64];
        if (has_acc) {
          tmem_ld64(t_addr + cc, v64);
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) v64[i] = 0.f;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = cc + 32 * h;
          if (c >= ncols) break;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = v64[32 * h + i];
          store_chunk<kPair == 1, kTF32>(v, ncols - c < 32 ? ncols - c : 32, col0 + c, drow, valid, p, o, lane, stg,
                                         rowd, bulk_live);
        }
      }
      // every lane's TMEM reads are complete; one arrival per warp hands the
      // accumulator back (the peer's go to the leader, whose MMA reuses both TMEMs)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty_bar(acc));
        else mbar_arrive_remote(map_to_rank(tempty_bar(acc), lead_rank));
      }
      if (++acc == nacc) { acc = 0; acc_phase ^= 1u; }
      if (signal >= 0) {
        pend = signal;
        pend_n += 1;
        pend_writes = pend_writes || signal_writes;
      }
    }
    flush();
    if (lane == 0) bulk_wait_all();   // bulk stores read shared memory until they complete
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kCG2) cluster_sync_all();   // no CTA leaves while another may signal it
  tc_fence_after();
  if (warp == 1) {
    if constexpr (kCG2)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                   : "memory");
  }
}

// ------------------------------------------------------------------ small kernels
struct RoundJob {
  int32_t n;
  const float *src[16];
  float *dst[16];
  int64_t count[16];
};

// Round fp32 inputs to the nearest tf32 value once, so the tensor cores see
// round-to-nearest operands rather than truncated ones.
__global__ void round_tf32_kernel(const __grid_constant__ RoundJob job) {
  for (int b = 0; b < job.n; ++b) {
    const float *s = job.src[b];
    float *d = job.dst[b];
    const int64_t n = job.count[b];
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t n4 = n / 4;
    const float4 *s4 = reinterpret_cast<const float4 *>(s);
    float4 *d4 = reinterpret_cast<float4 *>(d);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4; i += stride) {
      float4 x = s4[i];
      x.x = round_tf32(x.x); x.y = round_tf32(x.y); x.z = round_tf32(x.z); x.w = round_tf32(x.w);
      d4[i] = x;
    }
    for (int64_t i = 4 * n4 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n; i += stride)
      d[i] = round_tf32(s[i]);
  }
}

// Transposed, tf32-rounded copies of input views (TF32 tensor cores read
// K-major operands only). 256 threads: a 32 x 32 tile through shared memory,
// coalesced reads along the source's columns and writes along the copy's.
__global__ void transpose_round_kernel(const TJob *__restrict__ jobs, int njobs, int64_t ntiles) {
  __shared__ float tile[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    int lo = 0, hi = njobs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (jobs[mid].tile0 <= t) lo = mid; else hi = mid - 1;
    }
    const TJob J = jobs[lo];
    const int64_t local = t - J.tile0;
    const int64_t tr = (J.rows + 31) / 32;
    const int64_t r0 = (local % tr) * 32, c0 = (local / tr) * 32;
    for (int yy = ty; yy < 32; yy += 8) {
      const int64_t r = r0 + tx, c = c0 + yy;
      tile[yy][tx] = (r < J.rows && c < J.cols) ? J.src[r + c * J.src_ld] : 0.f;
    }
    __syncthreads();
    for (int yy = ty; yy < 32; yy += 8) {
      const int64_t c = c0 + tx, r = r0 + yy;
      if (r < J.rows && c < J.cols) J.dst[c + r * J.dst_ld] = round_tf32(tile[tx][yy]);
    }
    __syncthreads();
  }
}

// C <- beta * C (beta == 0: C <- 0 without reading C), column-major m x n.
__global__ void scale_c_kernel(float *C, int64_t ldc, int64_t m, int64_t n, float beta) {
  const int64_t total = m * n;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total; e += stride) {
    const int64_t r = e % m, c = e / m;
    float *x = C + r + c * ldc;
    *x = beta == 0.f ? 0.f : beta * *x;
  }
}

// A wait nothing will satisfy: exercises the bounded-wait path (test hook).
__global__ void unsatisfied_wait_kernel(const __grid_constant__ Params p) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bounded(smem_u32(&bar), 0, &abort_flag, p, 15);
  __syncthreads();
}

// ------------------------------------------------------------------ launchers
template <bool kTF32, int kPair>
cudaError_t launch_one(const Params &p, int grid, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(&tlr_task_gemm<kTF32, kPair>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if constexpr (kPair == 1) {
    tlr_task_gemm<kTF32, 1><<<grid, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair;   // 2: one CTA pair; 4: two pairs
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, &tlr_task_gemm<kTF32, kPair>, p);
  }
}

// Clusters (of kPair CTAs) that can be resident at once (all must be, since
// tasks are assigned to clusters in turn).
template <bool kTF32, int kPair>
int resident_clusters() {
  static int n = -1;
  if (n < 0) {
    cudaFuncSetAttribute(&tlr_task_gemm<kTF32, kPair>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kPair, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, &tlr_task_gemm<kTF32, kPair>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      c = 0;
    }
    n = c;
  }
  return n;
}

int max_resident_pairs(bool tf32) { return tf32 ? resident_clusters<true, 2>() : resident_clusters<false, 2>(); }
int max_resident_quads(bool tf32) { return tf32 ? resident_clusters<true, 4>() : resident_clusters<false, 4>(); }

cudaError_t launch_task_gemm(bool tf32, int pair, const Params &p, int grid, cudaStream_t stream) {
  if (pair == 4) return tf32 ? launch_one<true, 4>(p, grid, stream) : launch_one<false, 4>(p, grid, stream);
  if (pair == 2) return tf32 ? launch_one<true, 2>(p, grid, stream) : launch_one<false, 2>(p, grid, stream);
  return tf32 ? launch_one<true, 1>(p, grid, stream) : launch_one<false, 1>(p, grid, stream);
}

cudaError_t launch_round_tf32(const float *const *src, float *const *dst, const int64_t *count, int n,
                              int grid, cudaStream_t stream) {
  for (int b0 = 0; b0 < n; b0 += 16) {
    RoundJob job{};
    job.n = (n - b0) < 16 ? (n - b0) : 16;
    for (int b = 0; b < job.n; ++b) {
      job.src[b] = src[b0 + b];
      job.dst[b] = dst[b0 + b];
      job.count[b] = count[b0 + b];
    }
    round_tf32_kernel<<<grid, 256, 0, stream>>>(job);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_transpose_round(const TJob *jobs, int njobs, int64_t ntiles, int grid, cudaStream_t stream) {
  if (njobs <= 0 || ntiles <= 0) return cudaSuccess;
  transpose_round_kernel<<<grid, 256, 0, stream>>>(jobs, njobs, ntiles);
  return cudaGetLastError();
}

cudaError_t launch_scale_c(float *C, int64_t ldc, int64_t m, int64_t n, float beta, int grid,
                           cudaStream_t stream) {
  scale_c_kernel<<<grid, 256, 0, stream>>>(C, ldc, m, n, beta);
  return cudaGetLastError();
}

cudaError_t launch_unsatisfied_wait(const Params &p, cudaStream_t stream) {
  unsatisfied_wait_kernel<<<1, 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace tlr
