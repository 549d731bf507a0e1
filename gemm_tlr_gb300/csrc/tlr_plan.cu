// Host side of the Tile-Low-Rank GEMM library: descriptor validation, operand
// views, the rank-metadata planner, descriptor-table building and launches.
//
//   C <- alpha op(A) op(B) + beta C   ("Tile-Low-Rank GEMM: Designing Storage
//   Around the Contraction", opening section)
//
// Plan (same page, "Association order and workspace"): from ranks alone,
//   - rho_i / gamma_j (rank sums) give the final-stage costs of the two
//     association orders, F_R = sum_i 2 d_i W_J rho_i (U (S Z^T), one product
//     per tile row) and F_L = sum_j 2 d_j H_I gamma_j ((U S) Z^T, one per tile
//     column);
//   - C is split into rectangles of output tiles that fit the workspace:
//     widest feasible block of tile columns first, then the longest runs of tile
//     rows; each rectangle holds the full reduction over k and takes the cheaper
//     feasible order; rectangles run in sequence over one arena (two when one
//     launch overlaps the stages of consecutive rectangles).
// The left order is evaluated as the right order of the transposed product
// C^T = op(B)^T op(A)^T with a transposed store of the output tile, so both
// orders share one kernel path.
//
// Per rectangle three classes of tasks for the one task kernel (section "One
// product, three stages"):
//   L1  Stage 1 S_k = V_{:,k}^T W_{k,:} per contraction tile k (fused over i
//       and j), plus P_i = D_ii W_{i,:} (first half of D_A O_B) and the k=j block
//       V_ij^T D_jj of T_i (O_A D_B), both from "TLR Matrix Multiplication",
//       section "The easy terms";
//   L2  Stage 2 T_i[k-block, j-block] = S_ikj Z_kj^T, fused over i (rows of one
//       product scatter into the terminal matrices of several tile rows);
//   L3  Stage 3 C[i, J] = alpha (U_i T_i + P_ij Z_ij^T | D_ii D_ii) + beta C:
//       the sum over k is the tensor-core K-loop over the packed row panel U_i,
//       and the dense-diagonal terms are one more K segment of the same
//       accumulator, so every element of C is read and written once.
// One-TLR-operand products (dense B) skip Stage 2: L1 writes T_i rows
// V_{:,k}^T B_k directly, and L3 adds the segment D_ii B_i.
// Launches: with 256-wide final tiles, L1 and L2 of a rectangle run in one launch
// on single CTAs and L3 in the next on CTA pairs (L1 on pairs, in a launch of its
// own, for a product with a dense operand); otherwise one launch runs every
// class of every rectangle in order, L1-L2 of rectangle r + 1 mixed with L3 of
// r when there are two arenas.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <climits>
#include <functional>
#include <map>
#include <new>
#include <string>
#include <set>
#include <tuple>
#include <mutex>
#include <vector>

#include "tlr_gemm.h"
#include "tlr_tables.h"

namespace tlr {
cudaError_t launch_task_gemm(bool tf32, int pair, const Params &p, int grid, cudaStream_t stream);
int max_resident_pairs(bool tf32);
int max_resident_quads(bool tf32);
cudaError_t launch_round_tf32(const float *const *src, float *const *dst, const int64_t *count, int n,
                              int grid, cudaStream_t stream);
cudaError_t launch_scale_c(float *C, int64_t ldc, int64_t m, int64_t n, float beta, int grid,
                           cudaStream_t stream);
cudaError_t launch_transpose_round(const TJob *jobs, int njobs, int64_t ntiles, int grid, cudaStream_t stream);
cudaError_t launch_unsatisfied_wait(const Params &p, cudaStream_t stream);
}  // namespace tlr

using namespace tlr;

namespace {

constexpr int kKindStage1 = 0, kKindStage2 = 1, kKindStage3 = 2, kKindRound = 3, kKindScale = 4, kKindTasks = 5;
// launch classes of the two-launch-per-rectangle schedule
constexpr int kKindPrep = kKindStage2, kKindFinal = kKindStage3;
constexpr int kNumKinds = 6;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t align_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// ------------------------------------------------------------------ views
struct View {            // column-major matrix in device memory (elements)
  uint64_t addr = 0;
  int64_t rows = 0, cols = 0, ld = 0;
};

View sub_cols(const View &v, int64_t c0, int64_t c1, int es) {
  View s = v;
  s.addr = v.addr + static_cast<uint64_t>(c0 * v.ld * es);
  s.cols = c1 - c0;
  return s;
}

struct Part {            // contiguous run of one panel: tiles [t0, t1) of the panel index
  View v;                // d x (columns of the run)
  int t0 = 0, t1 = 0;
  int64_t col0 = 0;      // column of the run's first tile within the whole panel
};

// Stored TLR matrix (before op).
struct Stored {
  int ntr = 0, ntc = 0, m = 0;
  int64_t b = 0, brem = 0;
  bool boundary = false, diag_dense = false;
  std::vector<int64_t> rd, cd;
  std::vector<int32_t> rank;          // ntr*ntc, 0 on dense tiles
  std::vector<View> outer, inner;     // per low-rank tile
  std::vector<View> diag;             // per dense diagonal tile
  std::vector<std::vector<Part>> rowp, colp;
  std::vector<std::vector<int64_t>> rpos, cpos;   // tile column inside its row / col panel
  std::vector<int64_t> ucol, vcol;    // packed column offset of each low-rank tile in its buffer
};

// Logical operand op(X): either a TLR grid or a dense matrix.
struct LOp {
  bool dense = false;
  int nr = 0, nc = 0;
  std::vector<int64_t> rd, cd, ro, co;
  std::vector<int32_t> rank;
  std::vector<uint8_t> dtile;          // dense tile (diagonal) flag
  std::vector<View> outer, inner;      // op(X)_ik = outer inner^T
  std::vector<View> diag;              // stored dense tile behind op(X)_ii
  bool diag_trans = false;             // op(X)_ii = stored^T
  std::vector<std::vector<Part>> rowp, colp;
  std::vector<std::vector<int64_t>> rpos, cpos;
  View dv;                             // dense: stored matrix
  bool dtrans = false;                 // dense: op = T
  int32_t r(int i, int k) const { return rank[static_cast<size_t>(i) * nc + k]; }
  bool dt(int i, int k) const { return dtile[static_cast<size_t>(i) * nc + k] != 0; }
};

struct Operand {                       // validated descriptor plus device base addresses
  tlr_operand_t d;
  Stored s;
  int64_t u_elems = 0, v_elems = 0, d_elems = 0, buU = 0, buV = 0, bvU = 0, bvV = 0, g_elems = 0;
};

int elem_size(int dtype) { return dtype == TLR_F32 ? 4 : 2; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Compute stored geometry, packed offsets and the element count of each buffer.
tlr_status_t describe(const tlr_operand_t &d, Operand &o, bool check_pointers) {
  o.d = d;
  if (d.dtype != TLR_F32 && d.dtype != TLR_BF16 && d.dtype != TLR_F16) return TLR_STATUS_INVALID_ARG;
  if (d.rows <= 0 || d.cols <= 0) return TLR_STATUS_INVALID_ARG;
  const int es = elem_size(d.dtype);
  const int amod = 16 / es;
  if (d.kind == TLR_KIND_DENSE) {
    if (d.ld < d.rows) return TLR_STATUS_INVALID_ARG;
    if ((d.ld * es) % 16) return TLR_STATUS_ALIGNMENT;
    if (check_pointers) {
      if (!d.data) return TLR_STATUS_INVALID_ARG;
      if (!aligned16(d.data)) return TLR_STATUS_ALIGNMENT;
    }
    return TLR_STATUS_OK;
  }
  if (d.kind != TLR_KIND_TLR) return TLR_STATUS_INVALID_ARG;
  if (d.b <= 0 || !d.ranks) return TLR_STATUS_INVALID_ARG;
  Stored &s = o.s;
  s.b = d.b;
  s.diag_dense = d.diag_dense != 0;
  s.ntr = static_cast<int>(ceil_div(d.rows, d.b));
  s.ntc = static_cast<int>(ceil_div(d.cols, d.b));
  s.boundary = (d.rows % d.b) != 0 || (d.cols % d.b) != 0;
  if (s.diag_dense && d.rows != d.cols) return TLR_STATUS_INVALID_ARG;
  if (s.boundary && !s.diag_dense) return TLR_STATUS_UNSUPPORTED;
  s.m = s.boundary ? static_cast<int>(d.rows / d.b) : -1;
  s.brem = s.boundary ? d.rows - static_cast<int64_t>(s.m) * d.b : 0;
  if (s.boundary && s.m < 1) return TLR_STATUS_UNSUPPORTED;
  for (int i = 0; i < s.ntr; ++i) s.rd.push_back(std::min<int64_t>(d.b, d.rows - i * d.b));
  for (int k = 0; k < s.ntc; ++k) s.cd.push_back(std::min<int64_t>(d.b, d.cols - k * d.b));
  for (int64_t x : s.rd) if (x % amod) return TLR_STATUS_ALIGNMENT;
  for (int64_t x : s.cd) if (x % amod) return TLR_STATUS_ALIGNMENT;
  const size_t nt = static_cast<size_t>(s.ntr) * s.ntc;
  s.rank.assign(nt, 0);
  for (int i = 0; i < s.ntr; ++i)
    for (int k = 0; k < s.ntc; ++k) {
      if (s.diag_dense && i == k) continue;
      const int32_t r = d.ranks[static_cast<size_t>(i) * s.ntc + k];
      if (r < 0 || r > s.rd[i] || r > s.cd[k]) return TLR_STATUS_INVALID_ARG;
      s.rank[static_cast<size_t>(i) * s.ntc + k] = r;
    }
  auto R = [&](int i, int k) { return static_cast<int64_t>(s.rank[static_cast<size_t>(i) * s.ntc + k]); };
  auto lowrank = [&](int i, int k) { return !(s.diag_dense && i == k); };
  const int nr = s.boundary ? s.m : s.ntr, nc = s.boundary ? s.m : s.ntc;
  // packed column offsets (in factor columns)
  std::vector<int64_t> ucol(nt, -1), vcol(nt, -1);
  int64_t c = 0;
  for (int i = 0; i < nr; ++i)
    for (int k = 0; k < nc; ++k)
      if (lowrank(i, k)) { ucol[static_cast<size_t>(i) * s.ntc + k] = c; c += R(i, k); }
  const int64_t ucols = c;
  c = 0;
  for (int k = 0; k < nc; ++k)
    for (int i = 0; i < nr; ++i)
      if (lowrank(i, k)) { vcol[static_cast<size_t>(i) * s.ntc + k] = c; c += R(i, k); }
  int64_t bu_cols = 0, bv_cols = 0;
  if (s.boundary) {
    for (int i = 0; i < s.m; ++i) { ucol[static_cast<size_t>(i) * s.ntc + s.m] = bu_cols; vcol[static_cast<size_t>(i) * s.ntc + s.m] = bu_cols; bu_cols += R(i, s.m); }
    for (int j = 0; j < s.m; ++j) { ucol[static_cast<size_t>(s.m) * s.ntc + j] = bv_cols; vcol[static_cast<size_t>(s.m) * s.ntc + j] = bv_cols; bv_cols += R(s.m, j); }
  }
  o.u_elems = d.b * ucols;
  o.v_elems = d.b * ucols;
  o.d_elems = s.diag_dense ? static_cast<int64_t>(d.b) * d.b * nr : 0;
  o.buU = d.b * bu_cols;
  o.buV = s.brem * bu_cols;
  o.bvU = s.brem * bv_cols;
  o.bvV = d.b * bv_cols;
  o.g_elems = s.boundary ? s.brem * s.brem : 0;
  // optional caller offsets must agree with the prefix sums
  for (int i = 0; i < s.ntr; ++i)
    for (int k = 0; k < s.ntc; ++k) {
      if (!lowrank(i, k)) continue;
      const size_t t = static_cast<size_t>(i) * s.ntc + k;
      if (d.u_offsets && d.u_offsets[t] != s.rd[i] * ucol[t]) return TLR_STATUS_INVALID_ARG;
      if (d.v_offsets && d.v_offsets[t] != s.cd[k] * vcol[t]) return TLR_STATUS_INVALID_ARG;
    }
  if (check_pointers) {
    if ((ucols > 0) && (!d.U || !d.V)) return TLR_STATUS_INVALID_ARG;
    if (o.d_elems > 0 && !d.D) return TLR_STATUS_INVALID_ARG;
    if (bu_cols > 0 && (!d.bu_U || !d.bu_V)) return TLR_STATUS_INVALID_ARG;
    if (bv_cols > 0 && (!d.bv_U || !d.bv_V)) return TLR_STATUS_INVALID_ARG;
    if (s.boundary && !d.gamma) return TLR_STATUS_INVALID_ARG;
    for (const void *p : {d.U, d.V, d.D, d.bu_U, d.bu_V, d.bv_U, d.bv_V, d.gamma})
      if (p && !aligned16(p)) return TLR_STATUS_ALIGNMENT;
  }
  s.rpos.assign(s.ntr, std::vector<int64_t>(s.ntc, -1));
  s.cpos.assign(s.ntc, std::vector<int64_t>(s.ntr, -1));
  s.ucol = ucol;
  s.vcol = vcol;
  return TLR_STATUS_OK;
}

// Attach device addresses (possibly of rounded copies) to the stored views and
// build the row / column panels.
void bind(Operand &o, uint64_t U, uint64_t V, uint64_t D, uint64_t buU, uint64_t buV, uint64_t bvU,
          uint64_t bvV, uint64_t G) {
  Stored &s = o.s;
  const int es = elem_size(o.d.dtype);
  const int64_t b = s.b;
  const size_t nt = static_cast<size_t>(s.ntr) * s.ntc;
  const std::vector<int64_t> &ucol = s.ucol, &vcol = s.vcol;
  s.outer.assign(nt, View{});
  s.inner.assign(nt, View{});
  auto lowrank = [&](int i, int k) { return !(s.diag_dense && i == k); };
  for (int i = 0; i < s.ntr; ++i)
    for (int k = 0; k < s.ntc; ++k) {
      const size_t t = static_cast<size_t>(i) * s.ntc + k;
      if (!lowrank(i, k)) { s.outer[t] = View{}; s.inner[t] = View{}; continue; }
      const int64_t di = s.rd[i], dk = s.cd[k], r = s.rank[t];
      uint64_t ub = U, vb = V;
      if (s.boundary && k == s.m && i < s.m) { ub = buU; vb = buV; }
      else if (s.boundary && i == s.m && k < s.m) { ub = bvU; vb = bvV; }
      s.outer[t] = View{ub + static_cast<uint64_t>(di * ucol[t] * es), di, r, di};
      s.inner[t] = View{vb + static_cast<uint64_t>(dk * vcol[t] * es), dk, r, dk};
    }
  s.diag.assign(s.ntr, View{});
  if (s.diag_dense)
    for (int i = 0; i < s.ntr; ++i) {
      if (s.boundary && i == s.m) s.diag[i] = View{G, s.brem, s.brem, s.brem};
      else s.diag[i] = View{D + static_cast<uint64_t>(b * b * i * es), b, b, b};
    }
  // panels: a part is a run of consecutive tiles that share one buffer
  s.rowp.assign(s.ntr, {});
  s.colp.assign(s.ntc, {});
  for (int i = 0; i < s.ntr; ++i) {
    int64_t pos = 0;
    for (int k = 0; k < s.ntc; ++k) {
      if (!lowrank(i, k)) continue;
      const size_t t = static_cast<size_t>(i) * s.ntc + k;
      const View &v = s.outer[t];
      s.rpos[i][k] = pos;
      std::vector<Part> &P = s.rowp[i];
      const bool contiguous = !P.empty() &&
                              P.back().v.addr + static_cast<uint64_t>(P.back().v.cols * P.back().v.ld * es) == v.addr &&
                              P.back().v.ld == v.ld;
      if (contiguous) { P.back().v.cols += v.cols; P.back().t1 = k + 1; }
      else P.push_back(Part{View{v.addr, v.rows, v.cols, v.ld}, k, k + 1, pos});
      pos += v.cols;
    }
  }
  for (int k = 0; k < s.ntc; ++k) {
    int64_t pos = 0;
    for (int i = 0; i < s.ntr; ++i) {
      if (!lowrank(i, k)) continue;
      const size_t t = static_cast<size_t>(i) * s.ntc + k;
      const View &v = s.inner[t];
      s.cpos[k][i] = pos;
      std::vector<Part> &P = s.colp[k];
      const bool contiguous = !P.empty() &&
                              P.back().v.addr + static_cast<uint64_t>(P.back().v.cols * P.back().v.ld * es) == v.addr &&
                              P.back().v.ld == v.ld;
      if (contiguous) { P.back().v.cols += v.cols; P.back().t1 = i + 1; }
      else P.push_back(Part{View{v.addr, v.rows, v.cols, v.ld}, i, i + 1, pos});
      pos += v.cols;
    }
  }
}

// op(X) as a logical operand. Transposition swaps the factor families and the
// tile coordinates ("Tile-Low-Rank GEMM: Designing Storage Around the
// Contraction", section "Where fusion stops", paragraph "Transposes").
LOp logical(const Operand &o, bool trans, int64_t pseudo_b) {
  LOp L;
  if (o.d.kind == TLR_KIND_DENSE) {
    L.dense = true;
    L.dv = View{reinterpret_cast<uint64_t>(o.d.data), o.d.rows, o.d.cols, o.d.ld};
    L.dtrans = trans;
    const int64_t R = trans ? o.d.cols : o.d.rows, Cc = trans ? o.d.rows : o.d.cols;
    for (int64_t x = 0; x < R; x += pseudo_b) L.rd.push_back(std::min(pseudo_b, R - x));
    for (int64_t x = 0; x < Cc; x += pseudo_b) L.cd.push_back(std::min(pseudo_b, Cc - x));
  } else {
    const Stored &s = o.s;
    L.rd = trans ? s.cd : s.rd;
    L.cd = trans ? s.rd : s.cd;
    L.nr = trans ? s.ntc : s.ntr;
    L.nc = trans ? s.ntr : s.ntc;
    const size_t nt = static_cast<size_t>(L.nr) * L.nc;
    L.rank.assign(nt, 0);
    L.dtile.assign(nt, 0);
    L.outer.assign(nt, View{});
    L.inner.assign(nt, View{});
    for (int i = 0; i < L.nr; ++i)
      for (int k = 0; k < L.nc; ++k) {
        const int si = trans ? k : i, sk = trans ? i : k;
        const size_t st = static_cast<size_t>(si) * s.ntc + sk, lt = static_cast<size_t>(i) * L.nc + k;
        L.rank[lt] = s.rank[st];
        L.dtile[lt] = (s.diag_dense && si == sk) ? 1 : 0;
        L.outer[lt] = trans ? s.inner[st] : s.outer[st];
        L.inner[lt] = trans ? s.outer[st] : s.inner[st];
      }
    L.diag = s.diag;
    L.diag_trans = trans;
    L.rowp = trans ? s.colp : s.rowp;
    L.colp = trans ? s.rowp : s.colp;
    L.rpos = trans ? s.cpos : s.rpos;
    L.cpos = trans ? s.rpos : s.cpos;
  }
  L.nr = static_cast<int>(L.rd.size());
  L.nc = static_cast<int>(L.cd.size());
  L.ro.assign(L.nr + 1, 0);
  L.co.assign(L.nc + 1, 0);
  for (int i = 0; i < L.nr; ++i) L.ro[i + 1] = L.ro[i] + L.rd[i];
  for (int k = 0; k < L.nc; ++k) L.co[k + 1] = L.co[k] + L.cd[k];
  return L;
}

// Parts of a panel restricted to tiles [t0, t1): (sub-view, first tile, row offset in the result).
struct RPart {
  View v;
  std::vector<std::pair<int, int64_t>> tiles;   // (tile, column inside v)
  std::vector<int64_t> width;                   // rank of each listed tile
};

std::vector<RPart> restrict_panel(const std::vector<Part> &parts, const std::vector<int64_t> &pos,
                                  int t0, int t1, const std::function<int64_t(int)> &rank_of, int es) {
  std::vector<RPart> out;
  for (const Part &p : parts) {
    const int a = std::max(p.t0, t0), e = std::min(p.t1, t1);
    if (a >= e) continue;
    RPart rp;
    int64_t c0 = -1, c1 = -1;
    for (int t = a; t < e; ++t) {
      if (pos[t] < 0) continue;
      const int64_t r = rank_of(t);
      const int64_t local = pos[t] - p.col0;
      if (c0 < 0) c0 = local;
      c1 = local + r;
      rp.tiles.push_back({t, local});
      rp.width.push_back(r);
    }
    if (c0 < 0 || c1 <= c0) continue;
    rp.v = sub_cols(p.v, c0, c1, es);
    for (auto &tl : rp.tiles) tl.second -= c0;
    out.push_back(rp);
  }
  return out;
}

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

struct Rect {
  int i0, i1, j0, j1;
  bool left;
  bool triple = false;   // per-triple order (left ignored)
};

struct Launch {
  int kind;
  int64_t t0, t1;
  int pair = 1;          // CTAs per output tile in this launch (1, 2 for CTA pairs, 4 for two pairs sharing B)
  int bn = 0;            // output tile width of this launch's tasks (0: the plan's)
};

// ------------------------------------------------------------------ builder
using ViewKey = std::tuple<uint64_t, int64_t, int64_t, int64_t>;
ViewKey vkey(const View &v) { return std::make_tuple(v.addr, v.rows, v.cols, v.ld); }

struct ORef {           // an operand as the kernel reads it: tensor map + majorness
  int map = 0;
  bool mn = false;
};

struct Builder {
  const LOp &X;
  const LOp &Y;
  int es;
  bool tf32;
  int bn;
  bool trans_out;
  uint64_t ws;                          // arena base for this rectangle
  std::vector<CUtensorMap> *maps;
  std::map<std::tuple<uint64_t, int64_t, int64_t, int64_t, int>, int> *map_index;
  std::vector<Task> *tasks;
  std::vector<Seg> *segs;
  std::vector<Piece> *pieces;
  std::vector<Out> *outs;
  tlr_status_t status = TLR_STATUS_OK;
  double fl_s1 = 0, fl_s2 = 0, fl_s3 = 0, fl_dense = 0;
  double fl_launch[3] = {0, 0, 0};      // the same FLOPs by launch class
  bool dry = false;                     // validate only: no tensor maps are encoded
  bool f16 = false;                     // 16-bit operands and workspace are fp16 (else bf16)
  std::vector<std::pair<View, int>> *views = nullptr;   // every map's view and majorness
  // TF32 operands are read K-major only: a caller view that would be read
  // MN-major is replaced by its transposed copy (made by the pre-pass).
  const std::map<ViewKey, View> *tcopy = nullptr;
  std::set<ViewKey> *need_copy = nullptr;               // collection pass: record, do not build
  int bm = kBM;                         // output tile rows of the final products: 128, or 256 for a CTA pair
  int pair = 1;                         // CTAs per final-product tile (each epilogue warp of each signals)
  int prep_bm = kBM, prep_pair = 1;     // the same for Stages 1-2 and the dense precomputes
  int l1_bm = kBM, l1_pair = 1;         // Stage 1 and the dense precomputes (may run on pairs)
  int prep_bn = 256, l1_bn = 256;       // output tile widths of the Stage-2 and first-stage lists
  int cur_pair = 1;                     // of the list being built
  // Dependency counters of the merged launch (see Task in tlr_tables.h).
  std::vector<uint32_t> *counts = nullptr;              // signals each counter receives so far
  int32_t cS0 = -1, cPrep = -1, cL3 = -1;               // this rectangle's counters
  int32_t war = -1;                                     // counter of the rectangle whose arena we reuse
  uint32_t war_tgt = 0;
  int32_t sig = -1, sigw = 0, dep[2] = {-1, -1};
  uint32_t tgt[2] = {0, 0};
  void deps(int32_t s, int w, int32_t d0, int32_t d1) {
    sig = s;
    sigw = w;
    dep[0] = dep[1] = -1;
    tgt[0] = tgt[1] = 0;
    int n = 0;
    for (int32_t d : {d0, d1}) {
      if (d < 0) continue;
      const uint32_t t = d == war ? war_tgt : (counts ? (*counts)[d] : 0);
      if (t == 0) continue;
      dep[n] = d;
      tgt[n] = t;
      ++n;
    }
  }

  int map_of(const View &v, bool mn) {
    auto key = std::make_tuple(v.addr, v.rows, v.cols, v.ld, mn ? 1 : 0);
    auto it = map_index->find(key);
    if (it != map_index->end()) return it->second;
    CUtensorMap m;
    memset(&m, 0, sizeof m);
    if (views) views->push_back({v, mn ? 1 : 0});
    if (dry || need_copy) {
      const int idx = static_cast<int>(maps->size());
      maps->push_back(m);
      (*map_index)[key] = idx;
      return idx;
    }
    const int ch = 128 / es;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(v.rows), static_cast<cuuint64_t>(v.cols)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(v.ld * es)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(ch), static_cast<cuuint32_t>(mn ? ch : 64)};
    cuuint32_t estr[2] = {1, 1};
    auto fn = encode_fn();
    if (!fn || v.rows <= 0 || v.cols <= 0) { status = TLR_STATUS_CUDA_ERROR; return 0; }
    CUresult r = fn(&m, es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                : (f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16), 2,
                    reinterpret_cast<void *>(v.addr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { status = TLR_STATUS_CUDA_ERROR; return 0; }
    const int idx = static_cast<int>(maps->size());
    maps->push_back(m);
    (*map_index)[key] = idx;
    return idx;
  }

  // A caller-owned (input) view read with the given majorness.
  ORef input(const View &v, bool mn) {
    if (tf32 && mn) {
      if (need_copy) { need_copy->insert(vkey(v)); return ORef{map_of(v, true), true}; }
      auto it = tcopy ? tcopy->find(vkey(v)) : std::map<ViewKey, View>::const_iterator();
      if (!tcopy || it == tcopy->end()) { status = TLR_STATUS_UNSUPPORTED; return ORef{}; }
      return ORef{map_of(it->second, false), false};
    }
    return ORef{map_of(v, mn), mn};
  }
  // A workspace view (always produced K-major for the stage that reads it).
  ORef work(const View &v) { return ORef{map_of(v, false), false}; }

  // Rows [kk0, kk0+kl) x columns [n0, n0+nl) of a dense op(Y) as a B operand.
  ORef dense_block(int64_t kk0, int64_t kl, int64_t n0, int64_t nl) {
    const View &d = Y.dv;
    if (!Y.dtrans) return input(View{d.addr + static_cast<uint64_t>((kk0 + n0 * d.ld) * es), kl, nl, d.ld}, false);
    if (!tf32) return input(View{d.addr + static_cast<uint64_t>((n0 + kk0 * d.ld) * es), nl, kl, d.ld}, true);
    if (need_copy) { need_copy->insert(vkey(d)); return ORef{0, false}; }
    auto it = tcopy ? tcopy->find(vkey(d)) : std::map<ViewKey, View>::const_iterator();
    if (!tcopy || it == tcopy->end()) { status = TLR_STATUS_UNSUPPORTED; return ORef{}; }
    const View &c = it->second;   // stored^T: rows = stored cols (K), cols = stored rows (N)
    return ORef{map_of(View{c.addr + static_cast<uint64_t>((kk0 + n0 * c.ld) * es), kl, nl, c.ld}, false), false};
  }

  int out_ws(uint64_t ptr, int64_t ld, bool trans = false) {
    Out o;
    o.ptr = reinterpret_cast<void *>(ptr);
    o.ld = ld;
    o.kind = tf32 ? kOutTF32 : (f16 ? kOutF16 : kOutBF16);
    o.trans = trans ? 1 : 0;
    outs->push_back(o);
    return static_cast<int>(outs->size()) - 1;
  }
  int out_c() {
    Out o;
    o.ptr = nullptr;
    o.ld = 0;
    o.kind = kOutC;
    o.trans = trans_out ? 1 : 0;
    outs->push_back(o);
    return static_cast<int>(outs->size()) - 1;
  }
  void emit(int out, int64_t row0, int64_t col0, int64_t rows, int64_t cols, const std::vector<Seg> &sg,
            const std::vector<Piece> &pc) {
    Task t;
    memset(&t, 0, sizeof t);
    t.seg0 = static_cast<int32_t>(segs->size());
    t.nseg = static_cast<int32_t>(sg.size());
    t.out = out;
    t.rows = static_cast<int32_t>(rows);
    t.cols = static_cast<int32_t>(cols);
    t.piece0 = static_cast<int32_t>(pieces->size());
    t.npiece = static_cast<int32_t>(pc.size());
    t.row0 = row0;
    t.col0 = col0;
    t.signal = sig;
    t.signal_writes = sigw;
    t.dep[0] = dep[0];
    t.dep[1] = dep[1];
    t.dep_target[0] = tgt[0];
    t.dep_target[1] = tgt[1];
    if (sig >= 0 && counts) (*counts)[sig] += static_cast<uint32_t>(cur_pair * 4 * kEpiGroups);
    segs->insert(segs->end(), sg.begin(), sg.end());
    pieces->insert(pieces->end(), pc.begin(), pc.end());
    tasks->push_back(t);
  }
  static Seg seg(ORef a, ORef b, int64_t a_mn0, int64_t b_mn0, int64_t k_len) {
    Seg s;
    s.a_map = a.map;
    s.b_map = b.map;
    s.a_x = static_cast<int32_t>(a.mn ? a_mn0 : 0);
    s.a_y = static_cast<int32_t>(a.mn ? 0 : a_mn0);
    s.b_x = static_cast<int32_t>(b.mn ? b_mn0 : 0);
    s.b_y = static_cast<int32_t>(b.mn ? 0 : b_mn0);
    s.k_len = static_cast<int32_t>(k_len);
    s.flags = (a.mn ? kSegAMN : 0u) | (b.mn ? kSegBMN : 0u);
    return s;
  }
};

// Workspace layout of one rectangle (right order on X * Y).
//   S_k^T   (Gamma_k(J) padded) x sigma_k(I): Stage-1 output, the column block of
//           tile j starts on a 16-byte boundary so Stage 2 reads it K-major;
//   T       rows of T_i (parts padded to 8) x W_J columns; row-major for bf16
//           (a Stage-2 thread writes contiguous runs of one row, Stage 3 reads it
//           MN-major), column-major for tf32 (TF32 operands are read K-major);
//   P_i^T   (Gamma_i(J) padded) x d_i: (D_ii W_{i,J})^T, blocks aligned like S.
struct RectLayout {
  int i0, i1, j0, j1;
  int64_t WJ = 0;
  std::vector<int64_t> colT;                 // per j in [j0, j1]: column inside T / the C block
  std::vector<int64_t> Soff, Sld, Ssig;      // per k (Soff < 0: no S_k)
  std::vector<std::vector<int64_t>> Srow;    // per k, per j: first row of block j in S_k^T
  std::vector<int64_t> R;                    // per i: first T row
  std::vector<std::vector<int64_t>> Toff;    // per i, per part: first T row of the part
  int64_t Tld = 0, Toffset = 0;              // Tld: leading dimension of T's storage
  bool Trow = false;                         // T stored row-major (element (r, c) at c + r * Tld)
  int64_t Trows = 0;
  std::vector<int64_t> Poff, Pld;            // per i
  std::vector<std::vector<int64_t>> Prow;    // per i, per j
  int64_t bytes = 0;
};

RectLayout layout_rect(const LOp &X, const LOp &Y, int i0, int i1, int j0, int j1, int es) {
  RectLayout L;
  L.Trow = es == 2;
  L.i0 = i0; L.i1 = i1; L.j0 = j0; L.j1 = j1;
  L.colT.assign(j1 - j0 + 1, 0);
  for (int j = j0; j < j1; ++j) L.colT[j - j0 + 1] = L.colT[j - j0] + Y.cd[j];
  L.WJ = L.colT.back();
  int64_t off = 0;
  const int nk = X.nc;
  L.Soff.assign(nk, -1); L.Sld.assign(nk, 0); L.Ssig.assign(nk, 0); L.Srow.assign(nk, {});
  if (!Y.dense) {
    for (int k = 0; k < nk; ++k) {
      int64_t sig = 0;
      for (int i = i0; i < i1; ++i) if (!X.dt(i, k)) sig += X.r(i, k);
      L.Ssig[k] = sig;
      L.Srow[k].assign(j1 - j0, -1);
      int64_t g = 0;
      for (int j = j0; j < j1; ++j)
        if (!Y.dt(k, j) && Y.r(k, j) > 0) { L.Srow[k][j - j0] = g; g += align_up(Y.r(k, j), 8); }
      if (sig == 0 || g == 0) continue;
      L.Sld[k] = g;
      L.Soff[k] = off;
      off = align_up(off + g * sig * es, 256);
    }
  }
  L.R.assign(X.nr, 0);
  L.Toff.assign(X.nr, {});
  int64_t rows = 0;
  for (int i = i0; i < i1; ++i) {
    L.R[i] = rows;
    for (const Part &p : X.rowp[i]) {
      L.Toff[i].push_back(rows);
      rows += align_up(p.v.cols, 8);
    }
  }
  L.Trows = align_up(std::max<int64_t>(rows, 8), 8);
  L.Toffset = off;
  if (L.Trow) {
    L.Tld = align_up(L.WJ, 8);
    off = align_up(off + L.Trows * L.Tld * es, 256);
  } else {
    L.Tld = L.Trows;
    off = align_up(off + L.Tld * L.WJ * es, 256);
  }
  L.Poff.assign(X.nr, -1);
  L.Pld.assign(X.nr, 0);
  L.Prow.assign(X.nr, {});
  if (!Y.dense) {
    for (int i = i0; i < i1; ++i) {
      if (!(i < X.nc && X.dt(i, i))) continue;
      L.Prow[i].assign(j1 - j0, -1);
      int64_t g = 0;
      for (int j = j0; j < j1; ++j)
        if (!Y.dt(i, j) && Y.r(i, j) > 0) { L.Prow[i][j - j0] = g; g += align_up(Y.r(i, j), 8); }
      if (g == 0) continue;
      L.Pld[i] = g;
      L.Poff[i] = off;
      off = align_up(off + g * X.rd[i] * es, 256);
    }
  }
  L.bytes = off;
  return L;
}

// Final-stage cost of the right order on X * Y over a rectangle.
double final_cost(const LOp &X, int i0, int i1, int64_t WJ) {
  double f = 0;
  for (int i = i0; i < i1; ++i) {
    int64_t rho = 0;
    for (int k = 0; k < X.nc; ++k) if (!X.dt(i, k)) rho += X.r(i, k);
    f += 2.0 * static_cast<double>(X.rd[i]) * static_cast<double>(WJ) * static_cast<double>(rho);
  }
  return f;
}

// Row pieces of an output tile whose rows [w0, w0+rows) of a product's row
// space run over the tiles of `rp` (placed at row_base): each tile's rows go
// to dst_of(tile).
std::vector<Piece> pieces_for(const RPart &rp, int64_t row_base, int64_t w0, int64_t rows,
                              const std::function<int64_t(int)> &dst_of) {
  std::vector<Piece> pc;
  for (size_t q = 0; q < rp.tiles.size(); ++q) {
    const int64_t s = row_base + rp.tiles[q].second, e = s + rp.width[q];
    const int64_t a = std::max(s, w0), b = std::min(e, w0 + rows);
    if (a >= b) continue;
    Piece p;
    p.src0 = static_cast<int32_t>(a - w0);
    p.len = static_cast<int32_t>(b - a);
    p.dst0 = dst_of(rp.tiles[q].first) + (a - s);
    pc.push_back(p);
  }
  return pc;
}

// Build the tasks of one rectangle into the three launch lists.
void build_rect(Builder &B, const RectLayout &L, std::vector<Task> &l1, std::vector<Task> &l2,
                std::vector<Task> &l3) {
  const LOp &X = B.X;
  const LOp &Y = B.Y;
  const int es = B.es;
  int bn = B.l1_bn;                    // output tile width of the list being built
  int64_t BM = B.l1_bm;                // rows of an output tile (256 for a CTA pair)
  B.cur_pair = B.l1_pair;
  const int i0 = L.i0, i1 = L.i1, j0 = L.j0, j1 = L.j1;
  const uint64_t T = B.ws + static_cast<uint64_t>(L.Toffset);
  const int outT = B.out_ws(T, L.Tld, L.Trow);
  // T row of tile (i, k) of op(X)
  auto trow = [&](int i, int k) -> int64_t {
    const auto &parts = X.rowp[i];
    for (size_t pi = 0; pi < parts.size(); ++pi)
      if (k >= parts[pi].t0 && k < parts[pi].t1)
        return L.Toff[i][pi] + (X.rpos[i][k] - parts[pi].col0);
    return -1;
  };
  auto xcol = [&X](int k) { return [&X, k](int i) { return static_cast<int64_t>(X.r(i, k)); }; };
  auto yrow = [&Y](int k) { return [&Y, k](int j) { return static_cast<int64_t>(Y.r(k, j)); }; };

  // ---------------- L1: Stage 1, P, k=j blocks (or the dense-B product)
  B.tasks = &l1;
  for (int k = 0; k < X.nc; ++k) {
    std::vector<RPart> Ap = restrict_panel(X.colp[k], X.cpos[k], i0, i1, xcol(k), es);
    if (Ap.empty()) continue;
    B.deps(B.cPrep, 1, B.war, -1);
    if (Y.dense) {
      // T_i rows of block k: V_{:,k}^T B_k over the rectangle's columns
      const ORef bm = B.dense_block(Y.ro[k], Y.rd[k], Y.co[j0], L.WJ);
      for (const RPart &ap : Ap) {
        const ORef am = B.input(ap.v, false);
        for (int64_t mt = 0; mt < ceil_div(ap.v.cols, BM); ++mt) {
          const int64_t rows = std::min<int64_t>(BM, ap.v.cols - mt * BM);
          auto pc = pieces_for(ap, 0, mt * BM, rows, [&](int i) { return trow(i, k); });
          for (int64_t nt = 0; nt < ceil_div(L.WJ, bn); ++nt)
            B.emit(outT, 0, nt * bn, rows, std::min<int64_t>(bn, L.WJ - nt * bn),
                   {Builder::seg(am, bm, mt * BM, nt * bn, X.cd[k])}, pc);
        }
        B.fl_s1 += 2.0 * ap.v.cols * static_cast<double>(L.WJ) * X.cd[k];
      }
      continue;
    }
    // Stage 1, written transposed: S_k^T = W_{k,J}^T V_{k,I}
    if (L.Soff[k] >= 0) {
      B.deps(B.cS0 >= 0 ? B.cS0 + k : -1, 1, B.war, -1);
      const uint64_t S = B.ws + static_cast<uint64_t>(L.Soff[k]);
      const int outS = B.out_ws(S, L.Sld[k]);
      std::vector<RPart> Bp = restrict_panel(Y.rowp[k], Y.rpos[k], j0, j1, yrow(k), es);
      for (const RPart &bp : Bp) {
        const ORef am = B.input(bp.v, false);
        for (int64_t mt = 0; mt < ceil_div(bp.v.cols, BM); ++mt) {
          const int64_t rows = std::min<int64_t>(BM, bp.v.cols - mt * BM);
          auto pc = pieces_for(bp, 0, mt * BM, rows, [&](int j) { return L.Srow[k][j - j0]; });
          int64_t ra = 0;
          for (const RPart &ap : Ap) {
            const ORef bm = B.input(ap.v, false);
            for (int64_t nt = 0; nt < ceil_div(ap.v.cols, bn); ++nt)
              B.emit(outS, 0, ra + nt * bn, rows, std::min<int64_t>(bn, ap.v.cols - nt * bn),
                     {Builder::seg(am, bm, mt * BM, nt * bn, X.cd[k])}, pc);
            ra += ap.v.cols;
          }
        }
        for (const RPart &ap : Ap) B.fl_s1 += 2.0 * ap.v.cols * static_cast<double>(bp.v.cols) * X.cd[k];
      }
    }
    // k = j block with a dense tile of op(B): T_i[k-block, k-block] = V_ik^T D_kk
    if (k >= j0 && k < j1 && k < Y.nr && Y.dt(k, k)) {
      B.deps(B.cPrep, 1, B.war, -1);
      const ORef bm = B.input(Y.diag[k], Y.diag_trans);
      for (const RPart &ap : Ap) {
        const ORef am = B.input(ap.v, false);
        for (int64_t mt = 0; mt < ceil_div(ap.v.cols, BM); ++mt) {
          const int64_t rows = std::min<int64_t>(BM, ap.v.cols - mt * BM);
          auto pc = pieces_for(ap, 0, mt * BM, rows, [&](int i) { return trow(i, k); });
          for (int64_t nt = 0; nt < ceil_div(Y.cd[k], bn); ++nt)
            B.emit(outT, 0, L.colT[k - j0] + nt * bn, rows, std::min<int64_t>(bn, Y.cd[k] - nt * bn),
                   {Builder::seg(am, bm, mt * BM, nt * bn, Y.rd[k])}, pc);
        }
        B.fl_dense += 2.0 * ap.v.cols * static_cast<double>(Y.cd[k]) * Y.rd[k];
      }
    }
  }
  // P_i^T = (D_ii W_{i,J})^T = W_{i,J}^T D_ii^T, written transposed like S
  if (!Y.dense)
    for (int i = i0; i < i1; ++i) {
      if (L.Poff[i] < 0) continue;
      const uint64_t P = B.ws + static_cast<uint64_t>(L.Poff[i]);
      const int outP = B.out_ws(P, L.Pld[i]);
      B.deps(B.cPrep, 1, B.war, -1);
      // B operand (kk, n) = op(X)_ii[n, kk]: MN-major on the stored tile unless op(X)_ii is stored^T
      const ORef dm = B.input(X.diag[i], !X.diag_trans);
      std::vector<RPart> Bp = restrict_panel(Y.rowp[i], Y.rpos[i], j0, j1, yrow(i), es);
      for (const RPart &bp : Bp) {
        const ORef am = B.input(bp.v, false);
        for (int64_t mt = 0; mt < ceil_div(bp.v.cols, BM); ++mt) {
          const int64_t rows = std::min<int64_t>(BM, bp.v.cols - mt * BM);
          auto pc = pieces_for(bp, 0, mt * BM, rows, [&](int j) { return L.Prow[i][j - j0]; });
          for (int64_t nt = 0; nt < ceil_div(X.rd[i], bn); ++nt)
            B.emit(outP, 0, nt * bn, rows, std::min<int64_t>(bn, X.rd[i] - nt * bn),
                   {Builder::seg(am, dm, mt * BM, nt * bn, X.cd[i])}, pc);
        }
        B.fl_dense += 2.0 * X.rd[i] * static_cast<double>(bp.v.cols) * X.cd[i];
      }
    }

  B.fl_launch[0] += B.fl_s1 + B.fl_dense;
  const double before2 = B.fl_s2;
  // ---------------- L2: Stage 2, T_i[k, j] = S_ikj Z_kj^T fused over i
  B.tasks = &l2;
  BM = B.prep_bm;
  bn = B.prep_bn;
  B.cur_pair = B.prep_pair;
  if (!Y.dense)
    for (int k = 0; k < X.nc; ++k) {
      const int64_t sig = L.Ssig[k];
      if (sig == 0) continue;
      B.deps(B.cPrep, 1, B.cS0 >= 0 ? B.cS0 + k : -1, B.war);
      std::vector<RPart> Ap = restrict_panel(X.colp[k], X.cpos[k], i0, i1, xcol(k), es);
      std::vector<int64_t> base;
      int64_t acc = 0;
      for (const RPart &ap : Ap) { base.push_back(acc); acc += ap.v.cols; }
      for (int j = j0; j < j1; ++j) {
        if (Y.dt(k, j)) continue;                       // handled in L1
        const int64_t r = Y.r(k, j);
        ORef am, bm;
        if (r > 0) {
          am = B.work(View{B.ws + static_cast<uint64_t>(L.Soff[k] + L.Srow[k][j - j0] * es), r, sig, L.Sld[k]});
          bm = B.input(Y.inner[static_cast<size_t>(k) * Y.nc + j], true);
          B.fl_s2 += 2.0 * sig * static_cast<double>(Y.cd[j]) * r;
        }
        for (int64_t mt = 0; mt < ceil_div(sig, BM); ++mt) {
          const int64_t rows = std::min<int64_t>(BM, sig - mt * BM);
          std::vector<Piece> pc;
          for (size_t q = 0; q < Ap.size(); ++q) {
            auto pp = pieces_for(Ap[q], base[q], mt * BM, rows, [&](int i) { return trow(i, k); });
            pc.insert(pc.end(), pp.begin(), pp.end());
          }
          for (int64_t nt = 0; nt < ceil_div(Y.cd[j], bn); ++nt) {
            std::vector<Seg> sg;
            if (r > 0) sg.push_back(Builder::seg(am, bm, mt * BM, nt * bn, r));
            B.emit(outT, 0, L.colT[j - j0] + nt * bn, rows, std::min<int64_t>(bn, Y.cd[j] - nt * bn), sg, pc);
          }
        }
      }
    }

  B.fl_launch[1] += B.fl_s2 - before2;
  const double before3 = B.fl_s3 + B.fl_dense;
  // ---------------- L3: Stage 3, C[i, J] = alpha (U_i T_i + dense segment) + beta C
  B.tasks = &l3;
  BM = B.bm;
  bn = B.bn;
  B.cur_pair = B.pair;
  const int outC = B.out_c();
  B.deps(B.cL3, 0, B.cPrep, -1);
  for (int i = i0; i < i1; ++i) {
    const auto &parts = X.rowp[i];
    std::vector<ORef> am(parts.size()), bm(parts.size());
    int64_t rho = 0;
    for (size_t pi = 0; pi < parts.size(); ++pi) {
      if (parts[pi].v.cols <= 0) continue;
      am[pi] = B.input(parts[pi].v, true);
      if (L.Trow)   // MN-major B: view rows are T's columns (N), view columns its rows (K)
        bm[pi] = ORef{B.map_of(View{T + static_cast<uint64_t>(L.Toff[i][pi] * L.Tld * es), L.WJ, parts[pi].v.cols, L.Tld}, true), true};
      else
        bm[pi] = B.work(View{T + static_cast<uint64_t>(L.Toff[i][pi] * es), parts[pi].v.cols, L.WJ, L.Tld});
      rho += parts[pi].v.cols;
    }
    B.fl_s3 += 2.0 * X.rd[i] * static_cast<double>(L.WJ) * rho;
    const bool xdiag = i < X.nc && X.dt(i, i);
    ORef dm;
    if (xdiag) dm = B.input(X.diag[i], !X.diag_trans);
    for (int j = j0; j < j1; ++j) {
      ORef sa, sb;
      int64_t klen = 0;
      if (xdiag) {
        if (Y.dense) {
          sa = dm; sb = B.dense_block(Y.ro[i], Y.rd[i], Y.co[j], Y.cd[j]); klen = X.cd[i];
        } else if (j == i && Y.dt(i, i)) {
          sa = dm; sb = B.input(Y.diag[i], Y.diag_trans); klen = X.cd[i];
        } else if (!Y.dt(i, j) && Y.r(i, j) > 0) {
          klen = Y.r(i, j);
          sa = B.work(View{B.ws + static_cast<uint64_t>(L.Poff[i] + L.Prow[i][j - j0] * es), klen, X.rd[i], L.Pld[i]});
          sb = B.input(Y.inner[static_cast<size_t>(i) * Y.nc + j], true);
        }
        if (klen > 0) B.fl_dense += 2.0 * X.rd[i] * static_cast<double>(Y.cd[j]) * klen;
      }
      // Ticket order inside a block of kTicketBatch column tiles: row tile
      // first. A CTA claims kTicketBatch consecutive tickets, so it gets one row
      // tile (one slice of U_i) against kTicketBatch column tiles of T_i, and
      // the CTAs holding the other row tiles read the same T columns at the same
      // time, while they are in L2. (Consecutive row tiles of one column tile in
      // one batch made a CTA re-read that T chunk after L2 had dropped it.)
      const int64_t nnt = ceil_div(Y.cd[j], bn), nmt = ceil_div(X.rd[i], BM);
      for (int64_t nt0 = 0; nt0 < nnt; nt0 += kTicketBatch)
        for (int64_t mt = 0; mt < nmt; ++mt)
          for (int64_t nt = nt0; nt < std::min<int64_t>(nnt, nt0 + kTicketBatch); ++nt) {
          std::vector<Seg> sg;
          for (size_t pi = 0; pi < parts.size(); ++pi)
            if (parts[pi].v.cols > 0)
              sg.push_back(Builder::seg(am[pi], bm[pi], mt * BM, L.colT[j - j0] + nt * bn, parts[pi].v.cols));
          if (klen > 0) sg.push_back(Builder::seg(sa, sb, mt * BM, nt * bn, klen));
          B.emit(outC, X.ro[i] + mt * BM, Y.co[j] + nt * bn, std::min<int64_t>(BM, X.rd[i] - mt * BM),
                 std::min<int64_t>(bn, Y.cd[j] - nt * bn), sg, {});
        }
    }
  }
  B.fl_launch[2] += B.fl_s3 + B.fl_dense - before3;
}

// ------------------------------------------------------------------ per-triple order
// "TLR Matrix Multiplication", section "The O_A O_B terms": once the coupling
// product S_ikj = V_ik^T W_kj is formed, each tile triple (i, k, j) takes the
// cheaper of the two remaining contractions, decided by min(r_ik, r_kj):
//   right  T^R_ikj = S_ikj Z_kj^T (r_ik x d_j), then C_ij += U_ik T^R_ikj   (r_ik <= r_kj)
//   left   T^L_ikj = U_ik S_ikj   (d_i x r_kj), then C_ij += T^L_ikj Z_kj^T (r_kj <  r_ik)
// so the final product of a pair (i, j) runs over K = sum_k min(r_ik, r_kj)
// instead of rho_i (or gamma_j). The dense-tile terms take a fixed side: the
// k = j block V_ij^T D_jj is a right block (K = r_ij), the k = i block
// D_ii W_ij is a left block (P_ij, K = r_ij), and D_ii D_ii is a segment of its own.
//
// Storage (one rectangle of output tiles): the coupling products S_k^T as in the
// per-rectangle orders (one Stage-1 product per k, shared by both sides); the
// right blocks of a pair (i, j), in ascending k, form a matrix T^R_ij of
// sum r_ik rows and d_j columns, the left blocks (transposed, T^L_ikj^T, r_kj x d_i)
// a matrix T^L_ij; all of them are packed into two row-major buffers with one
// leading dimension, so nothing is stored for a block the pair does not use.
// Stage 2 of the right side is fused over i (one product per (k, j), rows of
// S_k^T for the tile rows that take the right side), that of the left side over j
// (one product per (k, i): T^L^T = S^T U_ik^T). The final product of a tile of C
// is one K-loop over the runs of consecutive right blocks (U_i panel against
// T^R_ij) and of left blocks (T^L_ij against the Z_j panel).
//
// A task's K-loop takes at most kMaxSegs operand segments. When the sides of a
// pair alternate so often that its runs need more, the run whose side change
// costs the fewest extra final-product FLOPs is given the other side, until the
// tile fits (never needed for rank maps that decay with |i - j|).

enum : uint8_t { kSideNone = 0, kSideRight = 1, kSideLeft = 2 };

struct TripleLayout {
  int i0 = 0, i1 = 0, j0 = 0, j1 = 0, nk = 0;
  std::vector<int64_t> Soff, Sld, Ssig;        // per k, as RectLayout
  std::vector<std::vector<int64_t>> Srow;      // per k, per j: first row of block j in S_k^T
  std::vector<uint8_t> side;                   // per (i, j, k): kSide*
  std::vector<int64_t> trow;                   // per (i, j, k): row of the block in its buffer, -1
  std::vector<int64_t> tR0, tRn, tL0, tLn;     // per (i, j): first row and rows of T^R_ij, T^L_ij
  int64_t ldT = 0, TRoff = 0, TLoff = 0, TRrows = 0, TLrows = 0;
  int64_t bytes = 0;
  size_t ij(int i, int j) const { return static_cast<size_t>(i - i0) * (j1 - j0) + (j - j0); }
  size_t ijk(int i, int j, int k) const { return ij(i, j) * nk + k; }
};

// Operand segments of the final product of pair (i, j) under `side`, in K-loop
// order: right runs over the U_i panel parts, then left runs over the Z_j panel
// parts. Each entry: (panel part view restricted to the run, first block k, run width).
struct TripleRun {
  bool right;
  View panel;          // U_i columns (right) or Z_j columns (left) of the run
  int k_first;
  int64_t width;
};

std::vector<TripleRun> triple_runs(const LOp &X, const LOp &Y, const TripleLayout &L, int i, int j, int es) {
  std::vector<TripleRun> out;
  // right: U_i panel, tiles k of op(A)'s row i in panel order
  for (const Part &p : X.rowp[i]) {
    bool open = false;
    int64_t c0 = 0, c1 = 0;
    int kf = -1;
    for (int k = p.t0; k < p.t1; ++k) {
      if (X.rpos[i][k] < 0) continue;
      const int64_t r = X.r(i, k);
      if (r == 0) continue;
      const bool in = L.side[L.ijk(i, j, k)] == kSideRight;
      const int64_t lc = X.rpos[i][k] - p.col0;
      if (in && !open) { open = true; c0 = lc; kf = k; }
      if (in) c1 = lc + r;
      if (!in && open) { out.push_back(TripleRun{true, sub_cols(p.v, c0, c1, es), kf, c1 - c0}); open = false; }
    }
    if (open) out.push_back(TripleRun{true, sub_cols(p.v, c0, c1, es), kf, c1 - c0});
  }
  // left: Z_j panel, tiles k of op(B)'s column j in panel order
  for (const Part &p : Y.colp[j]) {
    bool open = false;
    int64_t c0 = 0, c1 = 0;
    int kf = -1;
    for (int k = p.t0; k < p.t1; ++k) {
      if (Y.cpos[j][k] < 0) continue;
      const int64_t r = Y.r(k, j);
      if (r == 0) continue;
      const bool in = L.side[L.ijk(i, j, k)] == kSideLeft;
      const int64_t lc = Y.cpos[j][k] - p.col0;
      if (in && !open) { open = true; c0 = lc; kf = k; }
      if (in) c1 = lc + r;
      if (!in && open) { out.push_back(TripleRun{false, sub_cols(p.v, c0, c1, es), kf, c1 - c0}); open = false; }
    }
    if (open) out.push_back(TripleRun{false, sub_cols(p.v, c0, c1, es), kf, c1 - c0});
  }
  return out;
}

// Side of every (i, k, j) of the rectangle by min(r_ik, r_kj) (tie: right), the
// fixed sides of the dense-tile blocks, and the coarsening that keeps every
// output tile within kMaxSegs segments.
void triple_sides(const LOp &X, const LOp &Y, TripleLayout &L, int es) {
  const int nk = X.nc;
  L.side.assign(static_cast<size_t>(L.i1 - L.i0) * (L.j1 - L.j0) * nk, kSideNone);
  for (int i = L.i0; i < L.i1; ++i)
    for (int j = L.j0; j < L.j1; ++j) {
      for (int k = 0; k < nk; ++k) {
        uint8_t sd = kSideNone;
        if (X.dt(i, k)) {                       // k = i: D_ii B_ij
          if (!Y.dt(k, j) && Y.r(k, j) > 0) sd = kSideLeft;        // P_ij = D_ii W_ij
        } else if (Y.dt(k, j)) {                // k = j: A_ij D_jj
          if (X.r(i, k) > 0) sd = kSideRight;                       // V_ij^T D_jj
        } else if (X.r(i, k) > 0 && Y.r(k, j) > 0) {
          sd = X.r(i, k) <= Y.r(k, j) ? kSideRight : kSideLeft;
        }
        L.side[L.ijk(i, j, k)] = sd;
      }
      const bool dd = X.dt(i, i) && i < Y.nr && Y.dt(i, j);   // D_ii D_ii segment
      const size_t cap = static_cast<size_t>(kMaxSegs - (dd ? 1 : 0));
      std::vector<uint8_t> locked(nk, 0);                       // a block changes side at most once
      for (;;) {
        std::vector<TripleRun> runs = triple_runs(X, Y, L, i, j, es);
        if (runs.size() <= cap) break;
        // cheapest run to give the other side (dense-tile blocks keep theirs)
        double best = 1e300;
        int bk0 = -1, bk1 = -1;
        bool bright = true;
        for (const TripleRun &ru : runs) {
          // the run's blocks: consecutive ks from k_first covering `width` columns
          double extra = 0;
          int64_t w = 0;
          int k = ru.k_first, klast = ru.k_first;
          bool fixed = false;
          for (; k < nk && w < ru.width; ++k) {
            const uint8_t sd = L.side[L.ijk(i, j, k)];
            if (sd != (ru.right ? kSideRight : kSideLeft)) continue;
            if (X.dt(i, k) || Y.dt(k, j) || locked[k]) { fixed = true; break; }
            const int64_t ra = X.r(i, k), rb = Y.r(k, j);
            w += ru.right ? ra : rb;
            extra += 2.0 * static_cast<double>(X.rd[i]) * static_cast<double>(Y.cd[j]) *
                     static_cast<double>(ru.right ? rb - ra : ra - rb);
            klast = k;
          }
          if (fixed) continue;
          if (extra < best) { best = extra; bk0 = ru.k_first; bk1 = klast; bright = ru.right; }
        }
        if (bk0 < 0) {
          // nothing left to move run by run: one side for every block that can take
          // either (the cheaper one for the pair), which leaves a run per panel part
          double fr = 0, fl = 0;
          for (int k = 0; k < nk; ++k)
            if (!X.dt(i, k) && !Y.dt(k, j) && L.side[L.ijk(i, j, k)] != kSideNone) { fr += X.r(i, k); fl += Y.r(k, j); }
          for (int k = 0; k < nk; ++k)
            if (!X.dt(i, k) && !Y.dt(k, j) && L.side[L.ijk(i, j, k)] != kSideNone)
              L.side[L.ijk(i, j, k)] = fr <= fl ? kSideRight : kSideLeft;
          break;
        }
        for (int k = bk0; k <= bk1; ++k) {
          uint8_t &sd = L.side[L.ijk(i, j, k)];
          if (sd == (bright ? kSideRight : kSideLeft) && !X.dt(i, k) && !Y.dt(k, j)) {
            sd = bright ? kSideLeft : kSideRight;
            locked[k] = 1;
          }
        }
      }
    }
}

TripleLayout layout_triple(const LOp &X, const LOp &Y, int i0, int i1, int j0, int j1, int es) {
  TripleLayout L;
  L.i0 = i0; L.i1 = i1; L.j0 = j0; L.j1 = j1;
  L.nk = X.nc;
  const int nk = X.nc;
  int64_t off = 0;
  L.Soff.assign(nk, -1); L.Sld.assign(nk, 0); L.Ssig.assign(nk, 0); L.Srow.assign(nk, {});
  for (int k = 0; k < nk; ++k) {
    int64_t sig = 0;
    for (int i = i0; i < i1; ++i) if (!X.dt(i, k)) sig += X.r(i, k);
    L.Ssig[k] = sig;
    L.Srow[k].assign(j1 - j0, -1);
    int64_t g = 0;
    for (int j = j0; j < j1; ++j)
      if (!Y.dt(k, j) && Y.r(k, j) > 0) { L.Srow[k][j - j0] = g; g += align_up(Y.r(k, j), 8); }
    if (sig == 0 || g == 0) continue;
    L.Sld[k] = g;
    L.Soff[k] = off;
    off = align_up(off + g * sig * es, 256);
  }
  triple_sides(X, Y, L, es);
  int64_t dmax = 8;
  for (int j = j0; j < j1; ++j) dmax = std::max(dmax, Y.cd[j]);
  for (int i = i0; i < i1; ++i) dmax = std::max(dmax, X.rd[i]);
  L.ldT = align_up(dmax, 8);
  const size_t npair = static_cast<size_t>(i1 - i0) * (j1 - j0);
  L.tR0.assign(npair, 0); L.tRn.assign(npair, 0); L.tL0.assign(npair, 0); L.tLn.assign(npair, 0);
  L.trow.assign(npair * nk, -1);
  int64_t rr = 0, rl = 0;
  for (int i = i0; i < i1; ++i)
    for (int j = j0; j < j1; ++j) {
      const size_t q = L.ij(i, j);
      L.tR0[q] = rr;
      L.tL0[q] = rl;
      for (int k = 0; k < nk; ++k) {
        const uint8_t sd = L.side[L.ijk(i, j, k)];
        if (sd == kSideRight) { L.trow[L.ijk(i, j, k)] = rr; rr += X.r(i, k); }
        else if (sd == kSideLeft) { L.trow[L.ijk(i, j, k)] = rl; rl += Y.r(k, j); }
      }
      L.tRn[q] = rr - L.tR0[q];
      L.tLn[q] = rl - L.tL0[q];
      rr = align_up(rr, 8);
      rl = align_up(rl, 8);
    }
  L.TRrows = std::max<int64_t>(rr, 8);
  L.TLrows = std::max<int64_t>(rl, 8);
  L.TRoff = off;
  off = align_up(off + L.TRrows * L.ldT * es, 256);
  L.TLoff = off;
  off = align_up(off + L.TLrows * L.ldT * es, 256);
  L.bytes = off;
  return L;
}

void build_rect_triple(Builder &B, const TripleLayout &L, std::vector<Task> &l1, std::vector<Task> &l2,
                       std::vector<Task> &l3) {
  const LOp &X = B.X;
  const LOp &Y = B.Y;
  const int es = B.es;
  int bn = B.l1_bn;                    // output tile width of the list being built
  const int i0 = L.i0, i1 = L.i1, j0 = L.j0, j1 = L.j1, nk = L.nk;
  const uint64_t TR = B.ws + static_cast<uint64_t>(L.TRoff), TL = B.ws + static_cast<uint64_t>(L.TLoff);
  const int outR = B.out_ws(TR, L.ldT, true), outL = B.out_ws(TL, L.ldT, true);
  auto xcol = [&X](int k) { return [&X, k](int i) { return static_cast<int64_t>(X.r(i, k)); }; };
  auto yrow = [&Y](int k) { return [&Y, k](int j) { return static_cast<int64_t>(Y.r(k, j)); }; };
  int64_t BM = B.l1_bm;
  B.cur_pair = B.l1_pair;

  // ---------------- L1: Stage 1 (shared), V_ij^T D_jj into T^R, D_ii W_ij (transposed) into T^L
  B.tasks = &l1;
  for (int k = 0; k < nk; ++k) {
    std::vector<RPart> Ap = restrict_panel(X.colp[k], X.cpos[k], i0, i1, xcol(k), es);
    if (Ap.empty()) continue;
    if (L.Soff[k] >= 0) {
      B.deps(B.cS0 >= 0 ? B.cS0 + k : -1, 1, B.war, -1);
      const uint64_t S = B.ws + static_cast<uint64_t>(L.Soff[k]);
      const int outS = B.out_ws(S, L.Sld[k]);
      std::vector<RPart> Bp = restrict_panel(Y.rowp[k], Y.rpos[k], j0, j1, yrow(k), es);
      for (const RPart &bp : Bp) {
        const ORef am = B.input(bp.v, false);
        for (int64_t mt = 0; mt < ceil_div(bp.v.cols, BM); ++mt) {
          const int64_t rows = std::min<int64_t>(BM, bp.v.cols - mt * BM);
          auto pc = pieces_for(bp, 0, mt * BM, rows, [&](int j) { return L.Srow[k][j - j0]; });
          int64_t ra = 0;
          for (const RPart &ap : Ap) {
            const ORef bm = B.input(ap.v, false);
            for (int64_t nt = 0; nt < ceil_div(ap.v.cols, bn); ++nt)
              B.emit(outS, 0, ra + nt * bn, rows, std::min<int64_t>(bn, ap.v.cols - nt * bn),
                     {Builder::seg(am, bm, mt * BM, nt * bn, X.cd[k])}, pc);
            ra += ap.v.cols;
          }
        }
        for (const RPart &ap : Ap) B.fl_s1 += 2.0 * ap.v.cols * static_cast<double>(bp.v.cols) * X.cd[k];
      }
    }
    // k = j: T^R_ij block k=j = V_ij^T D_jj for the tile rows i of the rectangle
    if (k >= j0 && k < j1 && k < Y.nr && Y.dt(k, k)) {
      B.deps(B.cPrep, 1, B.war, -1);
      const ORef bm = B.input(Y.diag[k], Y.diag_trans);
      for (const RPart &ap : Ap) {
        const ORef am = B.input(ap.v, false);
        for (int64_t mt = 0; mt < ceil_div(ap.v.cols, BM); ++mt) {
          const int64_t rows = std::min<int64_t>(BM, ap.v.cols - mt * BM);
          auto pc = pieces_for(ap, 0, mt * BM, rows, [&](int i) { return L.trow[L.ijk(i, k, k)]; });
          for (int64_t nt = 0; nt < ceil_div(Y.cd[k], bn); ++nt)
            B.emit(outR, 0, nt * bn, rows, std::min<int64_t>(bn, Y.cd[k] - nt * bn),
                   {Builder::seg(am, bm, mt * BM, nt * bn, Y.rd[k])}, pc);
        }
        B.fl_dense += 2.0 * ap.v.cols * static_cast<double>(Y.cd[k]) * Y.rd[k];
      }
    }
  }
  // k = i: T^L_ij block k=i = (D_ii W_ij)^T = W_ij^T D_ii^T, for the tile columns j
  for (int i = i0; i < i1; ++i) {
    if (!(i < X.nc && X.dt(i, i))) continue;
    std::vector<RPart> Bp = restrict_panel(Y.rowp[i], Y.rpos[i], j0, j1, yrow(i), es);
    if (Bp.empty()) continue;
    B.deps(B.cPrep, 1, B.war, -1);
    const ORef dm = B.input(X.diag[i], !X.diag_trans);
    for (const RPart &bp : Bp) {
      const ORef am = B.input(bp.v, false);
      for (int64_t mt = 0; mt < ceil_div(bp.v.cols, BM); ++mt) {
        const int64_t rows = std::min<int64_t>(BM, bp.v.cols - mt * BM);
        auto pc = pieces_for(bp, 0, mt * BM, rows, [&](int j) { return L.trow[L.ijk(i, j, i)]; });
        for (int64_t nt = 0; nt < ceil_div(X.rd[i], bn); ++nt)
          B.emit(outL, 0, nt * bn, rows, std::min<int64_t>(bn, X.rd[i] - nt * bn),
                 {Builder::seg(am, dm, mt * BM, nt * bn, X.cd[i])}, pc);
      }
      B.fl_dense += 2.0 * X.rd[i] * static_cast<double>(bp.v.cols) * X.cd[i];
    }
  }
  B.fl_launch[0] += B.fl_s1 + B.fl_dense;

  // ---------------- L2: Stage 2 of both sides
  const double before2 = B.fl_s2;
  B.tasks = &l2;
  BM = B.prep_bm;
  bn = B.prep_bn;
  B.cur_pair = B.prep_pair;
  for (int k = 0; k < nk; ++k) {
    if (L.Soff[k] < 0) continue;
    const uint64_t S = B.ws + static_cast<uint64_t>(L.Soff[k]);
    B.deps(B.cPrep, 1, B.cS0 >= 0 ? B.cS0 + k : -1, B.war);
    std::vector<RPart> Ap = restrict_panel(X.colp[k], X.cpos[k], i0, i1, xcol(k), es);
    // rows of S_k^T's columns: tile row i of the rectangle at sigma position
    std::vector<std::pair<int, int64_t>> ipos;   // (i, column of block i in S_k^T)
    {
      int64_t acc = 0;
      for (const RPart &ap : Ap) {
        for (size_t q = 0; q < ap.tiles.size(); ++q) ipos.push_back({ap.tiles[q].first, acc + ap.tiles[q].second});
        acc += ap.v.cols;
      }
    }
    // right: per j, T^R rows S_ikj Z_kj^T for the i that take the right side (fused over i)
    for (int j = j0; j < j1; ++j) {
      if (Y.dt(k, j) || Y.r(k, j) <= 0) continue;
      const int64_t r = Y.r(k, j);
      // runs of consecutive tile rows (in S_k^T column order) on the right side
      std::vector<std::pair<int64_t, int64_t>> mr;   // [m0, m1) in S_k^T columns
      std::vector<std::vector<std::pair<int, int64_t>>> mi;
      for (auto &ip : ipos) {
        const int i = ip.first;
        const int64_t w = X.r(i, k);
        if (w == 0) continue;
        const bool in = L.side[L.ijk(i, j, k)] == kSideRight;
        if (!in) continue;
        if (!mr.empty() && mr.back().second == ip.second) { mr.back().second += w; mi.back().push_back(ip); }
        else { mr.push_back({ip.second, ip.second + w}); mi.push_back({ip}); }
      }
      if (mr.empty()) continue;
      const ORef am = B.work(View{S + static_cast<uint64_t>(L.Srow[k][j - j0] * es), r, L.Ssig[k], L.Sld[k]});
      const ORef bm = B.input(Y.inner[static_cast<size_t>(k) * Y.nc + j], true);
      for (size_t q = 0; q < mr.size(); ++q) {
        const int64_t m0 = mr[q].first, mlen = mr[q].second - mr[q].first;
        B.fl_s2 += 2.0 * mlen * static_cast<double>(Y.cd[j]) * r;
        for (int64_t mt = 0; mt < ceil_div(mlen, BM); ++mt) {
          const int64_t rows = std::min<int64_t>(BM, mlen - mt * BM);
          std::vector<Piece> pc;
          for (auto &ip : mi[q]) {
            const int64_t s = ip.second - m0, e = s + X.r(ip.first, k);
            const int64_t a = std::max(s, mt * BM), b2 = std::min(e, mt * BM + rows);
            if (a >= b2) continue;
            Piece pe;
            pe.src0 = static_cast<int32_t>(a - mt * BM);
            pe.len = static_cast<int32_t>(b2 - a);
            pe.dst0 = L.trow[L.ijk(ip.first, j, k)] + (a - s);
            pc.push_back(pe);
          }
          for (int64_t nt = 0; nt < ceil_div(Y.cd[j], bn); ++nt)
            B.emit(outR, 0, nt * bn, rows, std::min<int64_t>(bn, Y.cd[j] - nt * bn),
                   {Builder::seg(am, bm, m0 + mt * BM, nt * bn, r)}, pc);
        }
      }
    }
    // left: per i, T^L rows (U_ik S_ikj)^T = S_ikj^T U_ik^T for the j that take the left side (fused over j)
    for (auto &ip : ipos) {
      const int i = ip.first;
      const int64_t r = X.r(i, k);
      if (r == 0) continue;
      std::vector<std::pair<int64_t, int64_t>> mr;   // [m0, m1) in S_k^T rows
      std::vector<std::vector<int>> mj;
      for (int j = j0; j < j1; ++j) {
        if (Y.dt(k, j) || Y.r(k, j) <= 0) continue;
        if (L.side[L.ijk(i, j, k)] != kSideLeft) continue;
        const int64_t s = L.Srow[k][j - j0], e = s + Y.r(k, j);
        // consecutive S_k^T row blocks (padding rows between them are computed, not stored)
        if (!mr.empty() && align_up(mr.back().second, 8) == s) { mr.back().second = e; mj.back().push_back(j); }
        else { mr.push_back({s, e}); mj.push_back({j}); }
      }
      if (mr.empty()) continue;
      // A = S_k^T columns of block i, read MN-major (M = rows of S_k^T, K = r_ik)
      const ORef am = ORef{B.map_of(View{S + static_cast<uint64_t>(ip.second * L.Sld[k] * es), L.Sld[k], r, L.Sld[k]}, true), true};
      const ORef bm = B.input(X.outer[static_cast<size_t>(i) * X.nc + k], true);
      for (size_t q = 0; q < mr.size(); ++q) {
        const int64_t m0 = mr[q].first, mlen = mr[q].second - mr[q].first;
        for (int j : mj[q]) B.fl_s2 += 2.0 * Y.r(k, j) * static_cast<double>(X.rd[i]) * r;
        for (int64_t mt = 0; mt < ceil_div(mlen, BM); ++mt) {
          const int64_t rows = std::min<int64_t>(BM, mlen - mt * BM);
          std::vector<Piece> pc;
          for (int j : mj[q]) {
            const int64_t s = L.Srow[k][j - j0] - m0, e = s + Y.r(k, j);
            const int64_t a = std::max(s, mt * BM), b2 = std::min(e, mt * BM + rows);
            if (a >= b2) continue;
            Piece pe;
            pe.src0 = static_cast<int32_t>(a - mt * BM);
            pe.len = static_cast<int32_t>(b2 - a);
            pe.dst0 = L.trow[L.ijk(i, j, k)] + (a - s);
            pc.push_back(pe);
          }
          if (pc.empty()) continue;
          for (int64_t nt = 0; nt < ceil_div(X.rd[i], bn); ++nt)
            B.emit(outL, 0, nt * bn, rows, std::min<int64_t>(bn, X.rd[i] - nt * bn),
                   {Builder::seg(am, bm, m0 + mt * BM, nt * bn, r)}, pc);
        }
      }
    }
  }
  B.fl_launch[1] += B.fl_s2 - before2;

  // ---------------- L3: C[i, j] = alpha (right runs + left runs + D_ii D_ii) + beta C
  const double before3 = B.fl_s3 + B.fl_dense;
  B.tasks = &l3;
  BM = B.bm;
  bn = B.bn;
  B.cur_pair = B.pair;
  const int outC = B.out_c();
  B.deps(B.cL3, 0, B.cPrep, -1);
  for (int i = i0; i < i1; ++i)
    for (int j = j0; j < j1; ++j) {
      const size_t q = L.ij(i, j);
      std::vector<TripleRun> runs = triple_runs(X, Y, L, i, j, es);
      struct SegOps { ORef a, b; int64_t k; bool a_is_pair_rows; };
      std::vector<SegOps> ops;
      for (const TripleRun &ru : runs) {
        const int64_t row0 = L.trow[L.ijk(i, j, ru.k_first)];
        if (ru.right) {
          // A = U_i run (MN-major), B = T^R_ij rows (row-major: MN-major B)
          const ORef a = B.input(ru.panel, true);
          const ORef b = ORef{B.map_of(View{TR + static_cast<uint64_t>(row0 * L.ldT * es), Y.cd[j], ru.width, L.ldT}, true), true};
          ops.push_back(SegOps{a, b, ru.width, false});
        } else {
          // A = T^L_ij rows (transposed blocks: MN-major A), B = Z_j run (MN-major)
          const ORef a = ORef{B.map_of(View{TL + static_cast<uint64_t>(row0 * L.ldT * es), X.rd[i], ru.width, L.ldT}, true), true};
          const ORef b = B.input(ru.panel, true);
          ops.push_back(SegOps{a, b, ru.width, true});
        }
      }
      // FLOPs: every block of the pair (the k = i block counts as a dense-tile term)
      for (int k = 0; k < nk; ++k) {
        const uint8_t sd = L.side[L.ijk(i, j, k)];
        if (sd == kSideNone) continue;
        const double f = 2.0 * static_cast<double>(X.rd[i]) * static_cast<double>(Y.cd[j]) *
                         (sd == kSideRight ? X.r(i, k) : Y.r(k, j));
        if (X.dt(i, k)) B.fl_dense += f; else B.fl_s3 += f;
      }
      ORef da, db;
      int64_t dk = 0;
      if (X.dt(i, i) && i < Y.nr && Y.dt(i, j)) {
        da = B.input(X.diag[i], !X.diag_trans);
        db = B.input(Y.diag[i], Y.diag_trans);
        dk = X.cd[i];
        B.fl_dense += 2.0 * X.rd[i] * static_cast<double>(Y.cd[j]) * dk;
      }
      (void)q;
      const int64_t nnt = ceil_div(Y.cd[j], bn), nmt = ceil_div(X.rd[i], BM);
      for (int64_t nt0 = 0; nt0 < nnt; nt0 += kTicketBatch)
        for (int64_t mt = 0; mt < nmt; ++mt)
          for (int64_t nt = nt0; nt < std::min<int64_t>(nnt, nt0 + kTicketBatch); ++nt) {
            std::vector<Seg> sg;
            for (const SegOps &o : ops) sg.push_back(Builder::seg(o.a, o.b, mt * BM, nt * bn, o.k));
            if (dk > 0) sg.push_back(Builder::seg(da, db, mt * BM, nt * bn, dk));
            B.emit(outC, X.ro[i] + mt * BM, Y.co[j] + nt * bn, std::min<int64_t>(BM, X.rd[i] - mt * BM),
                   std::min<int64_t>(bn, Y.cd[j] - nt * bn), sg, {});
          }
    }
  B.fl_launch[2] += B.fl_s3 + B.fl_dense - before3;
}

// Sort a launch's tasks by decreasing K so the persistent CTAs finish together.
void sort_by_work(std::vector<Task> &v, const std::vector<Seg> &segs) {
  std::stable_sort(v.begin(), v.end(), [&](const Task &a, const Task &b) {
    int64_t ka = 0, kb = 0;
    for (int s = 0; s < a.nseg; ++s) ka += segs[a.seg0 + s].k_len;
    for (int s = 0; s < b.nseg; ++s) kb += segs[b.seg0 + s].k_len;
    return ka > kb;
  });
}

int device_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  }
  return n;
}

}  // namespace

// ------------------------------------------------------------------ handle / plan
struct tlr_handle_s {
  cudaStream_t stream = nullptr;
  int device = -1;                      // device current at tlr_create
  unsigned int *d_err = nullptr;
  bool timing = false;
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> ev_used;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev_free;
  double ms[kNumKinds] = {0, 0, 0, 0, 0};
  int64_t count[kNumKinds] = {0, 0, 0, 0, 0};
  unsigned long long wait_limit_ns = 2000000000ull;
};

struct tlr_plan_s {
  tlr_handle_t h = nullptr;
  bool tf32 = false;
  bool f16 = false;                       // 16-bit operands are fp16 (else bf16)
  int bn = 256;
  int pair = 1;
  int64_t Cm = 0, Cn = 0;                 // dimensions of C
  void *d_tables = nullptr;
  const void *d_maps = nullptr;
  const Task *d_tasks = nullptr;
  const Seg *d_segs = nullptr;
  const Piece *d_pieces = nullptr;
  const Out *d_outs = nullptr;
  std::vector<Launch> launches;
  std::vector<tlr_rect_t> rects;          // output rectangles in execution order
  std::vector<const float *> round_src;
  std::vector<float *> round_dst;
  std::vector<int64_t> round_n;
  const TJob *d_tjobs = nullptr;
  unsigned int *d_counters = nullptr;   // one ticket per launch, then the dependency counters
  size_t counters_bytes = 0;
  int ntjobs = 0;
  int64_t ttiles = 0;
  tlr_plan_info_t info{};
};

namespace {

struct ProblemViews {
  Operand A, B;
  bool dense_left = false, dense_right = false;
  int dtype = TLR_F32;
  int64_t Cm = 0, Cn = 0, K = 0;
  int64_t pseudo_b = 0;
};

tlr_status_t prepare(tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A, const tlr_operand_t *B,
                     ProblemViews &pv, bool check_pointers) {
  if (!A || !B) return TLR_STATUS_INVALID_ARG;
  if ((opA != TLR_OP_N && opA != TLR_OP_T) || (opB != TLR_OP_N && opB != TLR_OP_T)) return TLR_STATUS_INVALID_ARG;
  tlr_status_t st = describe(*A, pv.A, check_pointers);
  if (st) return st;
  st = describe(*B, pv.B, check_pointers);
  if (st) return st;
  if (A->dtype != B->dtype) return TLR_STATUS_UNSUPPORTED;
  pv.dtype = A->dtype;
  pv.dense_left = A->kind == TLR_KIND_DENSE;
  pv.dense_right = B->kind == TLR_KIND_DENSE;
  if (pv.dense_left && pv.dense_right) return TLR_STATUS_UNSUPPORTED;
  pv.Cm = opA == TLR_OP_T ? A->cols : A->rows;
  pv.K = opA == TLR_OP_T ? A->rows : A->cols;
  const int64_t Kb = opB == TLR_OP_T ? B->cols : B->rows;
  pv.Cn = opB == TLR_OP_T ? B->rows : B->cols;
  if (pv.K != Kb) return TLR_STATUS_INVALID_ARG;
  // contraction tiles must line up
  const tlr_operand_t *T = pv.dense_left ? B : A;
  pv.pseudo_b = T->b;
  if (!pv.dense_left && !pv.dense_right && A->b != B->b) return TLR_STATUS_UNSUPPORTED;
  return TLR_STATUS_OK;
}

// Base addresses used by the kernels (originals, or tf32-rounded copies in the workspace).
struct Bases { uint64_t a[8]; };

void collect_round(const Operand &o, bool tf32, uint64_t ws, int64_t &off, std::vector<const float *> &src,
                   std::vector<float *> &dst, std::vector<int64_t> &cnt, Bases &out) {
  const tlr_operand_t &d = o.d;
  const void *ptrs[8] = {d.U, d.V, d.D, d.bu_U, d.bu_V, d.bv_U, d.bv_V, d.gamma};
  const int64_t n[8] = {o.u_elems, o.v_elems, o.d_elems, o.buU, o.buV, o.bvU, o.bvV, o.g_elems};
  if (d.kind == TLR_KIND_DENSE) {
    const int64_t ne = d.ld * d.cols;
    if (tf32) {
      out.a[0] = ws + static_cast<uint64_t>(off);
      src.push_back(static_cast<const float *>(d.data)); dst.push_back(reinterpret_cast<float *>(out.a[0])); cnt.push_back(ne);
      off = align_up(off + ne * 4, 256);
    } else {
      out.a[0] = reinterpret_cast<uint64_t>(d.data);
    }
    return;
  }
  for (int b = 0; b < 8; ++b) {
    if (!tf32 || n[b] == 0) { out.a[b] = reinterpret_cast<uint64_t>(ptrs[b]); continue; }
    // the rounded copy's place is fixed even when sizing without buffers
    out.a[b] = ws + static_cast<uint64_t>(off);
    src.push_back(static_cast<const float *>(ptrs[b])); dst.push_back(reinterpret_cast<float *>(out.a[b])); cnt.push_back(n[b]);
    off = align_up(off + n[b] * 4, 256);
  }
}

struct TJobHost {
  uint64_t src, dst;
  int64_t src_ld, dst_ld, rows, cols;
};

struct PlanCore {
  ProblemViews pv;
  LOp XR, YR;     // right order:  op(A) * op(B)
  LOp XL, YL;     // left order:   op(B)^T * op(A)^T  (transposed output)
  bool can_right = true, can_left = true;
  int64_t fixed = 0;   // workspace taken by tf32-rounded and transposed input copies
  int nI = 0, nJ = 0;  // tile grid of C
  std::vector<int64_t> Crd, Ccd;
  std::vector<const float *> round_src;
  std::vector<float *> round_dst;
  std::vector<int64_t> round_n;
  std::map<ViewKey, View> tcopy;       // input view -> K-major transposed copy
  std::vector<TJobHost> tjobs;
};

void bind_operand(Operand &o, const Bases &b) {
  if (o.d.kind == TLR_KIND_DENSE) { o.d.data = reinterpret_cast<const void *>(b.a[0]); return; }
  bind(o, b.a[0], b.a[1], b.a[2], b.a[3], b.a[4], b.a[5], b.a[6], b.a[7]);
}

int choose_bn(const PlanCore &pc);
void build_rect(Builder &B, const RectLayout &L, std::vector<Task> &l1, std::vector<Task> &l2,
                std::vector<Task> &l3);

// TF32 products read every operand K-major. Find the input views some order
// would read MN-major (a dry build of the whole of C in each order) and give
// each a transposed copy after the rounded copies.
void collect_copies(PlanCore &pc, uint64_t ws) {
  std::set<ViewKey> need;
  const int es = elem_size(pc.pv.dtype);
  for (int order = 0; order < 2; ++order) {
    const bool left = order == 1;
    if ((left && !pc.can_left) || (!left && !pc.can_right)) continue;
    const LOp &X = left ? pc.XL : pc.XR;
    const LOp &Y = left ? pc.YL : pc.YR;
    std::vector<CUtensorMap> maps;
    std::map<std::tuple<uint64_t, int64_t, int64_t, int64_t, int>, int> mi;
    std::vector<Seg> segs;
    std::vector<Piece> pieces;
    std::vector<Out> outs;
    RectLayout L = layout_rect(X, Y, 0, X.nr, 0, Y.nc, es);
    Builder B{X, Y, es, true, choose_bn(pc), left, ws, &maps, &mi, nullptr, &segs, &pieces, &outs};
    B.dry = true;
    B.need_copy = &need;
    std::vector<Task> l1, l2, l3;
    build_rect(B, L, l1, l2, l3);
  }
  int64_t off = pc.fixed;
  for (const ViewKey &k : need) {
    const uint64_t addr = std::get<0>(k);
    const int64_t rows = std::get<1>(k), cols = std::get<2>(k), ld = std::get<3>(k);
    const int64_t dld = align_up(cols, 4);
    const uint64_t dst = ws + static_cast<uint64_t>(off);
    pc.tcopy[k] = View{dst, cols, rows, dld};
    pc.tjobs.push_back(TJobHost{addr, dst, ld, dld, rows, cols});
    off = align_up(off + dld * rows * 4, 256);
  }
  pc.fixed = off;
}

tlr_status_t core_init(PlanCore &pc, tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A,
                       const tlr_operand_t *B, bool check_pointers, uint64_t ws) {
  tlr_status_t st = prepare(opA, opB, A, B, pc.pv, check_pointers);
  if (st) return st;
  const bool tf32 = pc.pv.dtype == TLR_F32;
  Bases ba{}, bb{};
  int64_t off = 0;
  collect_round(pc.pv.A, tf32, ws, off, pc.round_src, pc.round_dst, pc.round_n, ba);
  collect_round(pc.pv.B, tf32, ws, off, pc.round_src, pc.round_dst, pc.round_n, bb);
  pc.fixed = off;
  bind_operand(pc.pv.A, ba);
  bind_operand(pc.pv.B, bb);
  const bool tA = opA == TLR_OP_T, tB = opB == TLR_OP_T;
  const int64_t pb = pc.pv.pseudo_b;
  pc.can_right = !pc.pv.dense_left;
  pc.can_left = !pc.pv.dense_right;
  if (pc.can_right) { pc.XR = logical(pc.pv.A, tA, pb); pc.YR = logical(pc.pv.B, tB, pb); }
  if (pc.can_left) { pc.XL = logical(pc.pv.B, !tB, pb); pc.YL = logical(pc.pv.A, !tA, pb); }
  if (pc.can_right) { pc.Crd = pc.XR.rd; pc.Ccd = pc.YR.cd; }
  else { pc.Crd = pc.YL.cd; pc.Ccd = pc.XL.rd; }
  pc.nI = static_cast<int>(pc.Crd.size());
  pc.nJ = static_cast<int>(pc.Ccd.size());
  if (tf32) collect_copies(pc, ws);
  return TLR_STATUS_OK;
}

// Workspace bytes of rectangle (rows [i0,i1), cols [j0,j1) of C) under an order.
// Workspace bytes of a per-triple rectangle (the right-order operands X = op(A), Y = op(B)).
int64_t rect_bytes_triple(const PlanCore &pc, int i0, int i1, int j0, int j1, int es) {
  return layout_triple(pc.XR, pc.YR, i0, i1, j0, j1, es).bytes;
}

// The per-triple order needs two TLR operands and a 16-bit element type (its
// left-side Stage 2 reads the coupling products MN-major).
bool can_triple(const PlanCore &pc) {
  return pc.can_right && pc.can_left && pc.pv.dtype != TLR_F32;
}

int64_t rect_bytes(const PlanCore &pc, int i0, int i1, int j0, int j1, bool left, int es) {
  if (!left) return layout_rect(pc.XR, pc.YR, i0, i1, j0, j1, es).bytes;
  return layout_rect(pc.XL, pc.YL, j0, j1, i0, i1, es).bytes;
}

double rect_cost(const PlanCore &pc, int i0, int i1, int j0, int j1, bool left) {
  if (!left) {
    int64_t W = 0;
    for (int j = j0; j < j1; ++j) W += pc.Ccd[j];
    return final_cost(pc.XR, i0, i1, W);
  }
  int64_t H = 0;
  for (int i = i0; i < i1; ++i) H += pc.Crd[i];
  return final_cost(pc.XL, j0, j1, H);
}

// Order for a rectangle: cheaper feasible one (tie: right); -1 if none fits.
int choose(const PlanCore &pc, int i0, int i1, int j0, int j1, int64_t arena, tlr_order_t force, int es) {
  if (force == TLR_ORDER_TRIPLE)
    return can_triple(pc) && rect_bytes_triple(pc, i0, i1, j0, j1, es) <= arena ? 2 : -1;
  const bool r_ok = pc.can_right && force != TLR_ORDER_LEFT && rect_bytes(pc, i0, i1, j0, j1, false, es) <= arena;
  const bool l_ok = pc.can_left && force != TLR_ORDER_RIGHT && rect_bytes(pc, i0, i1, j0, j1, true, es) <= arena;
  if (r_ok && l_ok) return rect_cost(pc, i0, i1, j0, j1, true) < rect_cost(pc, i0, i1, j0, j1, false) ? 1 : 0;
  if (r_ok) return 0;
  if (l_ok) return 1;
  return -1;
}

// Rectangles for a budget: widest feasible block of tile columns, then the
// longest runs of tile rows that fit.
bool split(const PlanCore &pc, int64_t arena, tlr_order_t force, int es, std::vector<Rect> &rects,
           int max_rows) {
  rects.clear();
  if (arena < 0) return false;
  int w = pc.nJ;
  for (; w >= 1; --w) {
    bool ok = true;
    for (int j0 = 0; ok && j0 < pc.nJ; j0 += w)
      for (int i = 0; ok && i < pc.nI; ++i)
        if (choose(pc, i, i + 1, j0, std::min(pc.nJ, j0 + w), arena, force, es) < 0) ok = false;
    if (ok) break;
  }
  if (w < 1) return false;
  for (int j0 = 0; j0 < pc.nJ; j0 += w) {
    const int j1 = std::min(pc.nJ, j0 + w);
    int i0 = 0;
    while (i0 < pc.nI) {
      int i1 = i0 + 1;
      while (i1 < pc.nI && (max_rows <= 0 || i1 - i0 < max_rows) &&
             choose(pc, i0, i1 + 1, j0, j1, arena, force, es) >= 0)
        ++i1;
      const int o = choose(pc, i0, i1, j0, j1, arena, force, es);
      rects.push_back(Rect{i0, i1, j0, j1, o == 1, o == 2});
      i0 = i1;
    }
  }
  return true;
}

// Largest rows per rectangle for a product large enough to pipeline: with at
// least four rectangles, Stages 1-2 of one rectangle run interleaved with
// Stage 3 of the previous one and only a quarter of the work is left without a
// partner at each end (measured best on the large workload: four rectangles
// beat two and eight). Small products keep one rectangle.
int pipeline_rows(const PlanCore &pc) {
  if (const char *e = getenv("TLR_PIPELINE_ROWS")) return atoi(e);   // tuning override (0: off)
  if (pc.nI < 8) return 0;
  const LOp &X = pc.can_right ? pc.XR : pc.XL;
  int64_t W = 0;
  for (int64_t x : pc.Ccd) W += x;
  if (final_cost(X, 0, X.nr, pc.can_right ? W : W) < 1e11) return 0;
  return static_cast<int>((pc.nI + 3) / 4);
}

// Rectangles and arena count for a budget. With more than one rectangle the
// arena is doubled so that rectangle r + 1 can be prepared while rectangle r
// finishes (the two-arena pipelining of the first page's "Association order
// and workspace"); a budget too small for two arenas runs the rectangles one
// after another in a single arena.
int choose_bn(const PlanCore &pc);
int choose_pair(const PlanCore &pc, int bn);

// CTAs per tile for Stages 1-2 and the dense precomputes. When the final
// products run on CTA pairs, the rest runs on single CTAs in a launch of its own
// before each rectangle's final products: Stage-2 tiles are short (K = one rank)
// and bound by their stores, and on the large bf16 product they ran 1.5x faster
// on single CTAs than on pairs (1.03 vs 1.53 ms), while the final products ran
// 1.2x faster on pairs (2.35 vs 2.85 ms); two launches per rectangle beat one
// merged launch of pairs. TLR_HYBRID=0 keeps the merged launch.
int choose_prep_pair(const PlanCore &pc, int bn, int pair) {
  (void)pc;
  (void)bn;
  if (pair != 2) return pair;
  if (const char *e = getenv("TLR_HYBRID"))
    if (atoi(e) == 0) return pair;
  return 1;
}

// CTAs per tile for Stage 1 and the dense precomputes when Stage 2 runs on
// single CTAs. A product with a dense operand has no Stage 2: its first-stage
// tiles (K = one tile of the contraction, 256 wide) run on CTA pairs, in a launch
// of their own before the final products (one TLR 16384^2 operand times a dense
// 16384 x 4096: 0.195 vs 0.243 ms for that launch). A TLR x TLR product keeps
// them with Stage 2 on single CTAs (large product: 0.49 ms on pairs in a launch
// of their own plus 0.85 for Stage 2, against 1.30 for the two together).
// TLR_L1_PAIR=0/1 overrides.
int choose_l1_pair(const PlanCore &pc, int prep_pair, int pair) {
  if (prep_pair == pair) return prep_pair;
  if (const char *e = getenv("TLR_L1_PAIR")) return atoi(e) == 1 ? pair : prep_pair;
  return (pc.pv.dense_left || pc.pv.dense_right) ? pair : prep_pair;
}

// Final-stage FLOPs of the per-triple order over all of C, on the same terms
// as F_R and F_L: each low-rank triple's K is min(r_ik, r_kj), the k = j block
// V_ij^T D_jj has K = r_ij, and the terms every order shares (D_ii W_ij Z_ij^T,
// D_ii D_ii) are left out; before any regrouping for the segment limit.
double triple_cost(const PlanCore &pc) {
  const LOp &X = pc.XR, &Y = pc.YR;
  double f = 0;
  for (int i = 0; i < X.nr; ++i)
    for (int j = 0; j < Y.nc; ++j) {
      const double dd = 2.0 * static_cast<double>(X.rd[i]) * static_cast<double>(Y.cd[j]);
      for (int k = 0; k < X.nc; ++k) {
        if (X.dt(i, k)) continue;
        if (Y.dt(k, j)) { f += dd * X.r(i, k); continue; }
        if (X.r(i, k) > 0 && Y.r(k, j) > 0) f += dd * std::min(X.r(i, k), Y.r(k, j));
      }
    }
  return f;
}

// TLR_ORDER_AUTO takes the per-triple order for the whole product when it is
// available and its final stage needs at most 90 % of the FLOPs of the cheaper
// single order (the large variable-rank product: 1.60e12 against 3.44e12
// FLOPs, 2.38 against 3.70 ms); otherwise the per-rectangle choice stays.
// TLR_TRIPLE=0/1 overrides (tuning).
tlr_order_t resolve_order(const PlanCore &pc, tlr_order_t order) {
  if (order != TLR_ORDER_AUTO) return order;
  if (!can_triple(pc)) return TLR_ORDER_PER_RECT;
  if (const char *e = getenv("TLR_TRIPLE")) return atoi(e) ? TLR_ORDER_TRIPLE : TLR_ORDER_PER_RECT;
  const double single = std::min(rect_cost(pc, 0, pc.nI, 0, pc.nJ, false), rect_cost(pc, 0, pc.nI, 0, pc.nJ, true));
  return triple_cost(pc) <= 0.9 * single ? TLR_ORDER_TRIPLE : TLR_ORDER_PER_RECT;
}

bool plan_split(const PlanCore &pc, int64_t budget, tlr_order_t force, int es, std::vector<Rect> &rects,
                int &narenas) {
  const int64_t avail = budget - pc.fixed;
  if (avail < 0) return false;
  force = resolve_order(pc, force);
  if (force == TLR_ORDER_TRIPLE && !can_triple(pc)) return false;
  {
    const int bn = choose_bn(pc), pair = choose_pair(pc, bn);
    if (choose_prep_pair(pc, bn, pair) != pair) {
      // Launches in stream order, so one arena. A large TLR x TLR product still
      // goes in at least four rectangles, whose smaller terminal matrices let
      // more of them take the cheaper association order (32768-wide bf16
      // product: 3.87 ms with four, 4.05 with two, 4.40 with eight); a product
      // with a dense operand (no Stage 2) takes the fewest the budget allows
      // (16384 x 16384 TLR times a dense 16384 x 4096: 0.54 ms in one, 0.66 in four).
      narenas = 1;
      const bool dense_operand = pc.pv.dense_left || pc.pv.dense_right;
      // per-triple plans also take the fewest rectangles (large product: 2.41 ms
      // in one, 2.64 in four): their terminal blocks are small and the order no
      // longer depends on the rectangle
      return split(pc, avail, force, es, rects, dense_operand || force == TLR_ORDER_TRIPLE ? 0 : pipeline_rows(pc));
    }
  }
  const int cap = pipeline_rows(pc);
  if (const char *e = getenv("TLR_ARENAS")) {                         // tuning override
    if (atoi(e) == 1) { narenas = 1; return split(pc, avail, force, es, rects, cap); }
  }
  if (cap == 0) {
    if (!split(pc, avail, force, es, rects, 0)) return false;
    narenas = 1;
    if (rects.size() == 1) return true;
    std::vector<Rect> two;
    if (split(pc, avail / 2, force, es, two, 0)) { rects = two; narenas = 2; }
    return true;
  }
  if (split(pc, avail / 2, force, es, rects, cap)) {
    narenas = rects.size() > 1 ? 2 : 1;
    return true;
  }
  narenas = 1;
  return split(pc, avail, force, es, rects, cap);
}

int64_t max_rect_bytes(const PlanCore &pc, const std::vector<Rect> &rects, int es) {
  int64_t m = 0;
  for (const Rect &r : rects)
    m = std::max(m, r.triple ? rect_bytes_triple(pc, r.i0, r.i1, r.j0, r.j1, es)
                             : rect_bytes(pc, r.i0, r.i1, r.j0, r.j1, r.left, es));
  return m;
}

// Output tile width: the smallest multiple of 64 covering a tile of C, at most 256.
int choose_bn(const PlanCore &pc) {
  int64_t bmax = 0;
  for (int64_t x : pc.Ccd) bmax = std::max(bmax, x);
  for (int64_t x : pc.Crd) bmax = std::max(bmax, x);
  return static_cast<int>(std::min<int64_t>(kMaxBN, align_up(std::max<int64_t>(bmax, 64), 64)));
}

// CTA pairs (256-row tiles, cta_group::2) need 256-wide tiles. A pair reads a
// third less operand data per FLOP than one CTA on a 128 x 256 tile and keeps
// six pipeline stages in the same shared memory, which the latency of the
// operand stream needs: measured on the 32768-wide bf16 product they are the
// faster choice overall although the T products alone run slower, and on large
// dense products they reach ~1.6 PFLOP/s against ~1.35 for single CTAs. One CTA
// per tile remains as an override (TLR_PAIR=1).
int choose_pair(const PlanCore &pc, int bn) {
  (void)pc;
  if (bn != kMaxBN) return 1;
  if (const char *e = getenv("TLR_PAIR")) return atoi(e) == 1 ? 1 : 2;
  return 2;
}

struct Tables {
  int bn = 256;
  int pair = 1;
  int prep_pair = 1;
  int l1_pair = 1;                          // Stage 1 and the dense precomputes
  int prep_bn = 256, l1_bn = 256;           // tile widths of the Stage-2 and first-stage lists
  std::vector<CUtensorMap> maps;
  std::map<std::tuple<uint64_t, int64_t, int64_t, int64_t, int>, int> map_index;
  std::vector<Task> all;
  std::vector<Seg> segs;
  std::vector<Piece> pieces;
  std::vector<Out> outs;
  std::vector<Launch> launches;
  std::vector<std::pair<View, int>> views;
  std::vector<int> task_rect;               // rectangle of each task
  std::vector<uint32_t> counter_counts;     // tasks signalling each dependency counter
  int narenas = 1;
  int64_t arena_bytes = 0;
  std::vector<uint64_t> rect_arena;         // arena base of each rectangle
  std::vector<RectLayout> layouts;          // per rectangle (in the order it was built)
  std::vector<uint8_t> rect_left;
  std::vector<uint8_t> rect_triple;
  std::vector<TripleLayout> tlayouts;       // per rectangle (empty unless per-triple)
  tlr_plan_info_t info{};
};

// Tile widths of the Stages 1-2 lists (tuning overrides TLR_PREP_BN and
// TLR_L1_BN, 128 or 256): on single CTAs in launches of their own a width of 128
// gives the kernel four accumulators instead of two. The lists keep the final
// products' width otherwise.
void choose_prep_widths(Tables &tb) {
  tb.prep_bn = tb.l1_bn = tb.bn;
  if (tb.bn != kMaxBN || tb.prep_pair != 1) return;
  if (const char *e = getenv("TLR_PREP_BN")) tb.prep_bn = atoi(e) == 128 ? 128 : kMaxBN;
  tb.l1_bn = tb.l1_pair == 1 ? tb.prep_bn : tb.bn;
  if (tb.l1_pair == 1)
    if (const char *e = getenv("TLR_L1_BN")) tb.l1_bn = atoi(e) == 128 ? 128 : kMaxBN;
}

// Estimated SM clocks of a task: tensor-core time or store time, whichever is larger.
double task_cost(const Task &t, const std::vector<Seg> &segs, const std::vector<Out> &outs, int bn) {
  int64_t k = 0;
  for (int q = 0; q < t.nseg; ++q) k += segs[t.seg0 + q].k_len;
  const double mma = static_cast<double>(bn) * static_cast<double>(k) / 32.0;
  const int ob = (outs[t.out].kind == kOutBF16 || outs[t.out].kind == kOutF16) ? 2 : 4;
  const double st = static_cast<double>(t.rows) * t.cols * ob / 32.0;
  return std::max(mma, st) + 200.0;
}

// Merge two task lists so that each list's share of the estimated work advances
// evenly; `from_a` records which list each merged task came from.
void interleave(const std::vector<Task> &a, const std::vector<Task> &b, const std::vector<Seg> &segs,
                const std::vector<Out> &outs, int bn, std::vector<Task> &out, std::vector<uint8_t> &from_a) {
  double ta = 0, tb = 0;
  for (const Task &t : a) ta += task_cost(t, segs, outs, bn);
  for (const Task &t : b) tb += task_cost(t, segs, outs, bn);
  size_t ia = 0, ib = 0;
  double ca = 0, cb = 0;
  while (ia < a.size() || ib < b.size()) {
    const bool take_a = ib >= b.size() || (ia < a.size() && ca / std::max(ta, 1.0) <= cb / std::max(tb, 1.0));
    if (take_a) { ca += task_cost(a[ia], segs, outs, bn); out.push_back(a[ia++]); from_a.push_back(1); }
    else { cb += task_cost(b[ib], segs, outs, bn); out.push_back(b[ib++]); from_a.push_back(0); }
  }
}

// Final-product tasks regrouped for clusters of two CTA pairs that share their
// B operand (the kernel's quad mode): groups of 2 x kTicketBatch tickets, the
// first kTicketBatch for the first pair and the rest for the second, slot q of
// one pair and slot q of the other with equal B-side segments. The builder
// emits a pair's batch as one row tile against up to kTicketBatch column tiles,
// and the next batch as the next row tile against the same column tiles, so
// consecutive batches pair up; a batch without a partner gets a copy of itself
// that stores nothing (rows = 0), and short batches are padded with tasks that
// have no segments and store nothing.
bool same_b_side(const Task &a, const Task &b, const std::vector<Seg> &segs) {
  if (a.nseg != b.nseg || a.cols != b.cols || a.col0 != b.col0) return false;
  for (int q = 0; q < a.nseg; ++q) {
    const Seg &x = segs[a.seg0 + q], &y = segs[b.seg0 + q];
    if (x.b_map != y.b_map || x.b_x != y.b_x || x.b_y != y.b_y || x.k_len != y.k_len || x.flags != y.flags) return false;
  }
  return true;
}

Task silent_copy(const Task &t, bool keep_segments) {
  Task n = t;
  n.rows = 0;
  if (!keep_segments) n.nseg = 0;
  n.signal = -1;
  n.signal_writes = 0;
  n.dep[0] = n.dep[1] = -1;
  n.dep_target[0] = n.dep_target[1] = 0;
  return n;
}

std::vector<Task> quad_regroup(const std::vector<Task> &fin, const std::vector<Seg> &segs) {
  std::vector<std::pair<size_t, size_t>> batches;
  for (size_t q = 0; q < fin.size();) {
    size_t e = q + 1;
    while (e < fin.size() && e - q < static_cast<size_t>(kTicketBatch) && fin[e].row0 == fin[q].row0 &&
           fin[e].out == fin[q].out)
      ++e;
    batches.push_back({q, e});
    q = e;
  }
  std::vector<Task> out;
  for (size_t bi = 0; bi < batches.size();) {
    const size_t a0 = batches[bi].first, n = batches[bi].second - a0;
    bool paired = bi + 1 < batches.size() && batches[bi + 1].second - batches[bi + 1].first == n;
    const size_t b0 = paired ? batches[bi + 1].first : 0;
    for (size_t k = 0; paired && k < n; ++k)
      if (!same_b_side(fin[a0 + k], fin[b0 + k], segs)) paired = false;
    for (size_t k = 0; k < static_cast<size_t>(kTicketBatch); ++k)
      out.push_back(k < n ? fin[a0 + k] : silent_copy(fin[a0], false));
    for (size_t k = 0; k < static_cast<size_t>(kTicketBatch); ++k) {
      if (k >= n) out.push_back(silent_copy(fin[a0], false));
      else out.push_back(paired ? fin[b0 + k] : silent_copy(fin[a0 + k], true));
    }
    bi += paired ? 2 : 1;
  }
  return out;
}

// Quad mode (two CTA pairs per cluster sharing B) for the final-product launches
// of the two-launch schedule. TLR_QUAD=0/1 overrides.
bool quad_enabled() {
  if (const char *e = getenv("TLR_QUAD")) return atoi(e) != 0;
  return false;
}

// Counters whose waiting tasks all run in later launches than every task that
// signals them: the kernel boundary already orders those stores before those
// reads, so the signals (and their fences) and the waits are dropped.
void drop_cross_launch_counters(Tables &tb) {
  const size_t nc = tb.counter_counts.size();
  if (nc == 0 || tb.launches.size() < 2) return;
  std::vector<int> launch_of(tb.all.size(), 0);
  for (size_t li = 0; li < tb.launches.size(); ++li)
    for (int64_t t = tb.launches[li].t0; t < tb.launches[li].t1; ++t) launch_of[t] = static_cast<int>(li);
  std::vector<int> last_sig(nc, -1), first_wait(nc, INT_MAX);
  for (size_t ti = 0; ti < tb.all.size(); ++ti) {
    const Task &t = tb.all[ti];
    if (t.signal >= 0) last_sig[t.signal] = std::max(last_sig[t.signal], launch_of[ti]);
    for (int d = 0; d < 2; ++d)
      if (t.dep[d] >= 0) first_wait[t.dep[d]] = std::min(first_wait[t.dep[d]], launch_of[ti]);
  }
  std::vector<uint8_t> keep(nc);
  for (size_t c = 0; c < nc; ++c) keep[c] = first_wait[c] <= last_sig[c];
  for (Task &t : tb.all) {
    if (t.signal >= 0 && !keep[t.signal]) { t.signal = -1; t.signal_writes = 0; }
    for (int d = 0; d < 2; ++d)
      if (t.dep[d] >= 0 && !keep[t.dep[d]]) { t.dep[d] = -1; t.dep_target[d] = 0; }
  }
  for (size_t c = 0; c < nc; ++c)
    if (!keep[c]) tb.counter_counts[c] = 0;
}

tlr_status_t build_tables(const PlanCore &pc, const std::vector<Rect> &rects, int narenas, uint64_t ws, bool dry,
                          Tables &tb) {
  const int es = elem_size(pc.pv.dtype);
  const bool tf32 = pc.pv.dtype == TLR_F32;
  const int64_t arena_bytes = align_up(max_rect_bytes(pc, rects, es), 256);
  tlr_plan_info_t &info = tb.info;
  memset(&info, 0, sizeof info);
  std::vector<std::vector<Task>> prep(rects.size()), fin(rects.size());
  std::vector<size_t> l2count(rects.size(), 0);
  std::vector<int32_t> cl3(rects.size(), -1);
  for (size_t ri = 0; ri < rects.size(); ++ri) {
    const Rect &r = rects[ri];
    const bool lft = r.left && !r.triple;
    const LOp &X = lft ? pc.XL : pc.XR;
    const LOp &Y = lft ? pc.YL : pc.YR;
    const int i0 = lft ? r.j0 : r.i0, i1 = lft ? r.j1 : r.i1;
    const int j0 = lft ? r.i0 : r.j0, j1 = lft ? r.i1 : r.j1;
    RectLayout L;
    TripleLayout TL3;
    if (r.triple) {
      TL3 = layout_triple(X, Y, i0, i1, j0, j1, es);
      if (TL3.TRrows >= INT32_MAX || TL3.TLrows >= INT32_MAX) return TLR_STATUS_UNSUPPORTED;
    } else {
      L = layout_rect(X, Y, i0, i1, j0, j1, es);
      if (L.Trows >= INT32_MAX) return TLR_STATUS_UNSUPPORTED;   // the epilogue holds T rows in 32 bits
    }
    const uint64_t arena = ws + static_cast<uint64_t>(pc.fixed + (static_cast<int64_t>(ri) % narenas) * arena_bytes);
    Builder B{X, Y, es, tf32, tb.bn, lft, arena, &tb.maps, &tb.map_index, nullptr, &tb.segs, &tb.pieces, &tb.outs};
    B.f16 = pc.pv.dtype == TLR_F16;
    B.dry = dry;
    B.views = &tb.views;
    B.tcopy = &pc.tcopy;
    B.pair = tb.pair;
    B.bm = kBM * tb.pair;
    B.prep_pair = tb.prep_pair;
    B.prep_bm = kBM * tb.prep_pair;
    B.l1_pair = tb.l1_pair;
    B.l1_bm = kBM * tb.l1_pair;
    B.prep_bn = tb.prep_bn;
    B.l1_bn = tb.l1_bn;
    // counters: S_k per contraction tile, "T and P ready", "Stage 3 done"
    B.counts = &tb.counter_counts;
    B.cS0 = static_cast<int32_t>(tb.counter_counts.size());
    tb.counter_counts.resize(tb.counter_counts.size() + X.nc, 0);
    B.cPrep = static_cast<int32_t>(tb.counter_counts.size());
    tb.counter_counts.push_back(0);
    // Stage 3 of this rectangle only signals when a later rectangle reuses its arena
    if (ri + narenas < rects.size()) {
      B.cL3 = static_cast<int32_t>(tb.counter_counts.size());
      tb.counter_counts.push_back(0);
    }
    cl3[ri] = B.cL3;
    if (ri >= static_cast<size_t>(narenas)) {
      B.war = cl3[ri - narenas];
      B.war_tgt = tb.counter_counts[B.war];
    }
    std::vector<Task> l1, l2, l3;
    if (r.triple) build_rect_triple(B, TL3, l1, l2, l3);
    else build_rect(B, L, l1, l2, l3);
    if (B.status) return B.status;
    l2count[ri] = l2.size();
    sort_by_work(l1, tb.segs);
    sort_by_work(l2, tb.segs);
    prep[ri] = l1;
    prep[ri].insert(prep[ri].end(), l2.begin(), l2.end());
    fin[ri] = l3;
    tb.layouts.push_back(L);
    tb.tlayouts.push_back(TL3);
    tb.rect_left.push_back(lft ? 1 : 0);
    tb.rect_triple.push_back(r.triple ? 1 : 0);
    tb.rect_arena.push_back(arena);
    info.runs += 1;
    if (r.triple) info.runs_triple += 1;
    else if (r.left) info.runs_left += 1;
    else info.runs_right += 1;
    info.flops_stage1 += B.fl_s1;
    info.flops_stage2 += B.fl_s2;
    info.flops_stage3 += B.fl_s3;
    info.flops_dense_terms += B.fl_dense;
    for (int q = 0; q < 3; ++q) info.flops_launch[q] += B.fl_launch[q];
    if (pc.can_right) info.flops_right_final += rect_cost(pc, r.i0, r.i1, r.j0, r.j1, false);
    if (pc.can_left) info.flops_left_final += rect_cost(pc, r.i0, r.i1, r.j0, r.j1, true);
  }
  // One launch; ticket order: the preparation of rectangle r (Stages 1-2) is
  // interleaved with Stage 3 of rectangle r - 1 when it has its own arena.
  std::vector<Task> stream;
  std::vector<int> stream_rect;
  auto push = [&](const std::vector<Task> &v, int rr) {
    for (const Task &t : v) { stream.push_back(t); stream_rect.push_back(rr); }
  };
  const size_t nr = rects.size();
  if (const char *e = getenv("TLR_SPLIT_LAUNCHES")) {
    // diagnostic: one launch per rectangle and stage class, in stream order
    if (atoi(e) == 1) {
      for (size_t ri = 0; ri < nr; ++ri) {
        const size_t n1 = prep[ri].size() - l2count[ri];
        std::vector<Task> a(prep[ri].begin(), prep[ri].begin() + n1), b(prep[ri].begin() + n1, prep[ri].end());
        const std::vector<Task> *lists[3] = {&a, &b, &fin[ri]};
        const int kinds[3] = {kKindStage1, kKindStage2, kKindStage3};
        const int pairs[3] = {tb.l1_pair, tb.prep_pair, tb.pair};
        for (int q = 0; q < 3; ++q) {
          if (lists[q]->empty()) continue;
          const int64_t t0 = static_cast<int64_t>(stream.size());
          push(*lists[q], static_cast<int>(ri));
          tb.launches.push_back(Launch{kinds[q], t0, static_cast<int64_t>(stream.size()), pairs[q]});
        }
      }
      tb.all = stream;
      tb.task_rect = stream_rect;
      drop_cross_launch_counters(tb);
      tb.narenas = narenas;
      tb.arena_bytes = arena_bytes;
      info.flops_executed = info.flops_stage1 + info.flops_stage2 + info.flops_stage3 + info.flops_dense_terms;
      info.tasks = static_cast<int64_t>(tb.all.size());
      return TLR_STATUS_OK;
    }
  }
  if (tb.prep_pair != tb.pair) {
    // Two launches per rectangle in stream order: Stages 1-2 and the dense
    // precomputes on single CTAs, then the final products on CTA pairs. A
    // launch only waits for counters of its own lower tickets; everything an
    // earlier launch signals is complete before the next one starts.
    for (size_t ri = 0; ri < nr; ++ri) {
      if (tb.l1_pair != tb.prep_pair || tb.l1_bn != tb.prep_bn) {   // Stage 1 and the dense precomputes in a launch of their own
        const size_t n1 = prep[ri].size() - l2count[ri];
        std::vector<Task> a(prep[ri].begin(), prep[ri].begin() + n1), b(prep[ri].begin() + n1, prep[ri].end());
        const std::vector<Task> *lists[3] = {&a, &b, &fin[ri]};
        const int kinds[3] = {kKindStage1, kKindPrep, kKindFinal}, pairs[3] = {tb.l1_pair, tb.prep_pair, tb.pair};
        const int bns[3] = {tb.l1_bn, tb.prep_bn, tb.bn};
        for (int q = 0; q < 3; ++q) {
          if (lists[q]->empty()) continue;
          const int64_t t0 = static_cast<int64_t>(stream.size());
          push(*lists[q], static_cast<int>(ri));
          tb.launches.push_back(Launch{kinds[q], t0, static_cast<int64_t>(stream.size()), pairs[q], bns[q]});
        }
        continue;
      }
      const bool quad = tb.pair == 2 && quad_enabled() && !fin[ri].empty();
      std::vector<Task> fq;
      if (quad) fq = quad_regroup(fin[ri], tb.segs);
      const std::vector<Task> *lists[2] = {&prep[ri], quad ? &fq : &fin[ri]};
      const int kinds[2] = {kKindPrep, kKindFinal}, pairs[2] = {tb.prep_pair, quad ? 4 : tb.pair};
      const int bns[2] = {tb.prep_bn, tb.bn};
      for (int q = 0; q < 2; ++q) {
        if (lists[q]->empty()) continue;
        const int64_t t0 = static_cast<int64_t>(stream.size());
        push(*lists[q], static_cast<int>(ri));
        tb.launches.push_back(Launch{kinds[q], t0, static_cast<int64_t>(stream.size()), pairs[q], bns[q]});
      }
    }
    tb.all = stream;
    tb.task_rect = stream_rect;
    drop_cross_launch_counters(tb);
    tb.narenas = narenas;
    tb.arena_bytes = arena_bytes;
    info.flops_executed = info.flops_stage1 + info.flops_stage2 + info.flops_stage3 + info.flops_dense_terms;
    info.tasks = static_cast<int64_t>(tb.all.size());
    return TLR_STATUS_OK;
  }
  for (size_t ri = 0; ri < nr; ++ri) {
    if (narenas >= 2 && ri >= 1) {
      std::vector<Task> mix;
      std::vector<uint8_t> from_a;
      interleave(prep[ri], fin[ri - 1], tb.segs, tb.outs, tb.bn, mix, from_a);
      for (size_t q = 0; q < mix.size(); ++q) {
        stream.push_back(mix[q]);
        stream_rect.push_back(static_cast<int>(from_a[q] ? ri : ri - 1));
      }
    } else {
      if (ri >= 1) push(fin[ri - 1], static_cast<int>(ri - 1));
      push(prep[ri], static_cast<int>(ri));
    }
  }
  if (nr) push(fin[nr - 1], static_cast<int>(nr - 1));
  tb.all = stream;
  tb.task_rect = stream_rect;
  tb.launches.push_back(Launch{kKindTasks, 0, static_cast<int64_t>(tb.all.size()), tb.pair});
  tb.narenas = narenas;
  tb.arena_bytes = arena_bytes;
  info.flops_executed = info.flops_stage1 + info.flops_stage2 + info.flops_stage3 + info.flops_dense_terms;
  info.tasks = static_cast<int64_t>(tb.all.size());
  return TLR_STATUS_OK;
}

// Rectangles as the ABI reports them: tile ranges of C and the order used.
std::vector<tlr_rect_t> abi_rects(const std::vector<Rect> &rects) {
  std::vector<tlr_rect_t> out;
  for (const Rect &r : rects) {
    tlr_rect_t x;
    x.i0 = r.i0; x.i1 = r.i1; x.j0 = r.j0; x.j1 = r.j1;
    x.order = r.triple ? TLR_ORDER_TRIPLE : (r.left ? TLR_ORDER_LEFT : TLR_ORDER_RIGHT);
    out.push_back(x);
  }
  return out;
}

tlr_status_t copy_rects(const std::vector<tlr_rect_t> &v, tlr_rect_t *rects, int32_t capacity, int32_t *count) {
  if (!count || capacity < 0 || (capacity > 0 && !rects)) return TLR_STATUS_INVALID_ARG;
  *count = static_cast<int32_t>(v.size());
  for (int32_t q = 0; q < capacity && q < *count; ++q) rects[q] = v[q];
  return TLR_STATUS_OK;
}

// ------------------------------------------------------------------ table validation
// Host-side proof that a plan's launches stay inside their buffers: every
// tensor-map view lies in one input buffer or the workspace, every segment's K
// range fits its views, every task writes inside its output, the tiles of C are
// covered exactly once, and in each rectangle the T rows Stage 3 reads are
// written exactly once by the earlier launches.
struct Region { uint64_t base; int64_t bytes; };

bool inside(const std::vector<Region> &regs, uint64_t a, int64_t n) {
  for (const Region &r : regs)
    if (a >= r.base && a + static_cast<uint64_t>(n) <= r.base + static_cast<uint64_t>(r.bytes)) return true;
  return false;
}

std::string validate_tables(const PlanCore &pc, const Tables &tb, uint64_t ws, int64_t ws_bytes) {
  const int es = elem_size(pc.pv.dtype);
  std::vector<Region> regs;
  regs.push_back(Region{ws, ws_bytes});
  for (const Operand *o : {&pc.pv.A, &pc.pv.B}) {
    if (o->d.kind == TLR_KIND_DENSE) { regs.push_back(Region{reinterpret_cast<uint64_t>(o->d.data), o->d.ld * o->d.cols * es}); continue; }
    const Stored &s = o->s;
    for (size_t t = 0; t < s.outer.size(); ++t) {
      if (s.outer[t].cols > 0) regs.push_back(Region{s.outer[t].addr, s.outer[t].ld * s.outer[t].cols * es});
      if (s.inner[t].cols > 0) regs.push_back(Region{s.inner[t].addr, s.inner[t].ld * s.inner[t].cols * es});
    }
    for (const Part &p : std::vector<Part>()) (void)p;
    for (const auto &P : s.rowp) for (const Part &p : P) regs.push_back(Region{p.v.addr, p.v.ld * p.v.cols * es});
    for (const auto &P : s.colp) for (const Part &p : P) regs.push_back(Region{p.v.addr, p.v.ld * p.v.cols * es});
    for (const View &v : s.diag) if (v.rows > 0) regs.push_back(Region{v.addr, v.ld * v.cols * es});
  }
  char buf[256];
  const bool tf32 = pc.pv.dtype == TLR_F32;
  for (size_t q = 0; q < pc.tjobs.size(); ++q) {
    const TJobHost &j = pc.tjobs[q];
    if (!inside(regs, j.src, ((j.cols - 1) * j.src_ld + j.rows) * es) ||
        j.dst < ws || j.dst + static_cast<uint64_t>(j.dst_ld * j.rows * es) > ws + static_cast<uint64_t>(pc.fixed)) {
      snprintf(buf, sizeof buf, "transposed copy %zu outside its buffers", q);
      return buf;
    }
  }
  for (size_t m = 0; m < tb.views.size(); ++m) {
    const View &v = tb.views[m].first;
    if (tf32 && tb.views[m].second) { snprintf(buf, sizeof buf, "map %zu: TF32 operand read MN-major", m); return buf; }
    if (v.rows <= 0 || v.cols <= 0 || v.ld < v.rows || (v.ld * es) % 16 || (v.addr & 15u)) {
      snprintf(buf, sizeof buf, "map %zu: bad view rows=%lld cols=%lld ld=%lld", m, (long long)v.rows, (long long)v.cols, (long long)v.ld);
      return buf;
    }
    const int64_t span = ((v.cols - 1) * v.ld + v.rows) * es;
    if (!inside(regs, v.addr, span)) { snprintf(buf, sizeof buf, "map %zu: view outside every buffer", m); return buf; }
  }
  const int64_t Cm = pc.pv.Cm, Cn = pc.pv.Cn;
  std::vector<int> task_pair(tb.all.size(), tb.pair), task_launch(tb.all.size(), 0);
  std::vector<uint8_t> task_quad(tb.all.size(), 0);
  std::vector<int> task_bn(tb.all.size(), tb.bn);
  for (size_t li = 0; li < tb.launches.size(); ++li) {
    const Launch &l = tb.launches[li];
    for (int64_t ti = l.t0; ti < l.t1; ++ti) {
      task_pair[ti] = l.pair == 4 ? 2 : l.pair;   // CTAs working on one task
      task_quad[ti] = l.pair == 4;
      task_bn[ti] = l.bn > 0 ? l.bn : tb.bn;
      task_launch[ti] = static_cast<int>(li);
    }
    if (l.pair == 4) {   // whole groups whose two halves agree slot by slot on B
      const int64_t g = 2 * kTicketBatch;
      if ((l.t1 - l.t0) % g) return "quad launch: not whole groups of tickets";
      for (int64_t t = l.t0; t < l.t1; t += g)
        for (int q = 0; q < kTicketBatch; ++q)
          if (!same_b_side(tb.all[t + q], tb.all[t + kTicketBatch + q], tb.segs)) {
            snprintf(buf, sizeof buf, "quad launch: tickets %lld and %lld differ in B", (long long)(t + q),
                     (long long)(t + kTicketBatch + q));
            return buf;
          }
    }
  }
  std::set<std::pair<int64_t, int64_t>> ctiles;
  double carea = 0;
  for (size_t ti = 0; ti < tb.all.size(); ++ti) {
    const Task &t = tb.all[ti];
    if (t.rows < (task_quad[ti] ? 0 : 1) || t.rows > kBM * task_pair[ti] || t.cols < 1 || t.cols > task_bn[ti] ||
        t.nseg > kMaxSegs) {
      snprintf(buf, sizeof buf, "task %zu: bad extent or segment count", ti);
      return buf;
    }
    if (t.rows == 0) {   // a quad launch's silent task: reads like its partner, stores nothing
      if (t.signal >= 0 || t.dep[0] >= 0 || t.dep[1] >= 0) { snprintf(buf, sizeof buf, "task %zu: silent task with counters", ti); return buf; }
    }
    for (int q = 0; q < t.nseg; ++q) {
      const Seg &g = tb.segs[t.seg0 + q];
      if (g.k_len <= 0 || g.a_map < 0 || g.b_map < 0 || g.a_map >= (int)tb.views.size() || g.b_map >= (int)tb.views.size()) {
        snprintf(buf, sizeof buf, "task %zu seg %d: bad map or K", ti, q); return buf;
      }
      const bool amn = g.flags & kSegAMN, bmn = g.flags & kSegBMN;
      if (tb.views[g.a_map].second != (amn ? 1 : 0) || tb.views[g.b_map].second != (bmn ? 1 : 0)) {
        snprintf(buf, sizeof buf, "task %zu seg %d: majorness differs from the map's box", ti, q); return buf;
      }
      const View &va = tb.views[g.a_map].first, &vb = tb.views[g.b_map].first;
      const int64_t aK = amn ? va.cols : va.rows, aMN = amn ? va.rows : va.cols;
      const int64_t bK = bmn ? vb.cols : vb.rows, bMN = bmn ? vb.rows : vb.cols;
      const int64_t a0 = amn ? g.a_x : g.a_y, b0 = bmn ? g.b_x : g.b_y;
      const int64_t ak = amn ? g.a_y : g.a_x, bk = bmn ? g.b_y : g.b_x;
      if (ak != 0 || bk != 0 || g.k_len > aK || g.k_len > bK) { snprintf(buf, sizeof buf, "task %zu seg %d: K range", ti, q); return buf; }
      if (a0 < 0 || a0 >= aMN || b0 < 0 || b0 >= bMN) { snprintf(buf, sizeof buf, "task %zu seg %d: tile outside its operand", ti, q); return buf; }
      if (((amn ? g.a_x : g.a_x) * es) % 16 || ((bmn ? g.b_x : g.b_x) * es) % 16) { snprintf(buf, sizeof buf, "task %zu seg %d: TMA x not 16-byte aligned", ti, q); return buf; }
    }
    const Out &o = tb.outs[t.out];
    if (o.kind == kOutC) {
      const int64_t R = o.trans ? Cn : Cm, Cc = o.trans ? Cm : Cn;
      if (t.npiece || t.row0 < 0 || t.col0 < 0 || t.row0 + t.rows > R || t.col0 + t.cols > Cc) {
        snprintf(buf, sizeof buf, "task %zu: C tile outside C", ti); return buf;
      }
      if (t.rows > 0 && !ctiles.insert({o.trans ? t.col0 : t.row0, o.trans ? t.row0 : t.col0}).second) {
        snprintf(buf, sizeof buf, "task %zu: C tile written twice", ti); return buf;
      }
      carea += static_cast<double>(t.rows) * t.cols;
    } else {
      const uint64_t base = reinterpret_cast<uint64_t>(o.ptr);
      int64_t rmin = INT64_MAX, rmax = -1;
      if (t.npiece == 0) { rmin = t.row0; rmax = t.row0 + t.rows - 1; }
      for (int q = 0; q < t.npiece; ++q) {
        const Piece &pe = tb.pieces[t.piece0 + q];
        if (pe.src0 < 0 || pe.len <= 0 || pe.src0 + pe.len > t.rows) { snprintf(buf, sizeof buf, "task %zu: bad piece", ti); return buf; }
        rmin = std::min<int64_t>(rmin, pe.dst0);
        rmax = std::max<int64_t>(rmax, pe.dst0 + pe.len - 1);
      }
      uint64_t lo, hi;
      if (o.trans) {   // element (r, c) at c + r * ld
        if (rmin < 0 || t.col0 < 0 || t.col0 + t.cols > o.ld) { snprintf(buf, sizeof buf, "task %zu: column beyond the leading dimension", ti); return buf; }
        lo = base + static_cast<uint64_t>((t.col0 + rmin * o.ld) * es);
        hi = base + static_cast<uint64_t>((t.col0 + t.cols + rmax * o.ld) * es);
      } else {
        if (rmin < 0 || rmax >= o.ld) { snprintf(buf, sizeof buf, "task %zu: row beyond the leading dimension", ti); return buf; }
        lo = base + static_cast<uint64_t>((rmin + t.col0 * o.ld) * es);
        hi = base + static_cast<uint64_t>((rmax + (t.col0 + t.cols - 1) * o.ld + 1) * es);
      }
      if (lo < ws + static_cast<uint64_t>(pc.fixed) || hi > ws + static_cast<uint64_t>(ws_bytes)) {
        snprintf(buf, sizeof buf, "task %zu: workspace write outside the arena", ti); return buf;
      }
    }
  }
  if (carea != static_cast<double>(Cm) * static_cast<double>(Cn)) return "tiles of C do not cover C exactly";
  // dependencies: every counter a task waits for reaches its target only through
  // tasks with lower tickets, and the target is the number of signalling tasks
  {
    const size_t nc = tb.counter_counts.size();
    std::vector<int64_t> last(nc, -1);
    std::vector<uint32_t> cnt(nc, 0);
    for (size_t ti = 0; ti < tb.all.size(); ++ti) {
      const Task &t = tb.all[ti];
      for (int d = 0; d < 2; ++d) {
        if (t.dep[d] < 0) continue;
        if (static_cast<size_t>(t.dep[d]) >= nc) { snprintf(buf, sizeof buf, "task %zu: bad counter", ti); return buf; }
        // every wait is met inside its own launch (counters are not reset between launches,
        // but a wait whose signals all came from earlier launches would only cost time)
        if (last[t.dep[d]] < 0 || task_launch[last[t.dep[d]]] != task_launch[ti]) {
          snprintf(buf, sizeof buf, "task %zu: waits for counter %d, last signalled outside its launch", ti, t.dep[d]);
          return buf;
        }
        if (t.dep_target[d] != tb.counter_counts[t.dep[d]] || cnt[t.dep[d]] != t.dep_target[d]) {
          snprintf(buf, sizeof buf, "task %zu: waits for counter %d before all %u signals have lower tickets",
                   ti, t.dep[d], t.dep_target[d]);
          return buf;
        }
      }
      if (t.signal >= 0) {
        if (static_cast<size_t>(t.signal) >= nc) { snprintf(buf, sizeof buf, "task %zu: bad signal", ti); return buf; }
        cnt[t.signal] += static_cast<uint32_t>(task_pair[ti] * 4 * kEpiGroups);
        last[t.signal] = static_cast<int64_t>(ti);
      }
    }
    for (size_t c = 0; c < nc; ++c)
      if (cnt[c] != tb.counter_counts[c]) return "counter counts differ";
  }
  // per-triple rectangles: every terminal-buffer element a final product reads
  // was written exactly once (by the launches before it)
  for (size_t ri = 0; ri < tb.layouts.size(); ++ri) {
    if (!tb.rect_triple[ri]) continue;
    const TripleLayout &L = tb.tlayouts[ri];
    const uint64_t bufs[2] = {tb.rect_arena[ri] + static_cast<uint64_t>(L.TRoff),
                              tb.rect_arena[ri] + static_cast<uint64_t>(L.TLoff)};
    const int64_t nrows[2] = {L.TRrows, L.TLrows};
    const int64_t rowb = L.ldT * es;
    std::vector<std::vector<std::pair<int32_t, int32_t>>> wr[2];
    for (int q = 0; q < 2; ++q) wr[q].assign(static_cast<size_t>(nrows[q]), {});
    std::vector<size_t> finals;
    for (size_t ti = 0; ti < tb.all.size(); ++ti) {
      if (tb.task_rect[ti] != static_cast<int>(ri)) continue;
      const Task &t = tb.all[ti];
      const Out &o = tb.outs[t.out];
      if (o.kind == kOutC) { finals.push_back(ti); continue; }
      const uint64_t base = reinterpret_cast<uint64_t>(o.ptr);
      const int q = base == bufs[0] ? 0 : (base == bufs[1] ? 1 : -1);
      if (q < 0) continue;
      auto add = [&](int64_t r0, int64_t n) {
        for (int64_t r = r0; r < r0 + n; ++r)
          if (r >= 0 && r < nrows[q]) wr[q][r].push_back({static_cast<int32_t>(t.col0), static_cast<int32_t>(t.col0 + t.cols)});
      };
      if (t.npiece == 0) add(t.row0, t.rows);
      for (int pq = 0; pq < t.npiece; ++pq) add(tb.pieces[t.piece0 + pq].dst0, tb.pieces[t.piece0 + pq].len);
    }
    for (int q = 0; q < 2; ++q)
      for (auto &v : wr[q]) {
        std::sort(v.begin(), v.end());
        for (size_t x = 1; x < v.size(); ++x)
          if (v[x].first < v[x - 1].second) { snprintf(buf, sizeof buf, "rect %zu: terminal element written twice", ri); return buf; }
      }
    auto covered = [&](int q, int64_t r, int64_t c0, int64_t c1) {
      if (r < 0 || r >= nrows[q]) return false;
      int64_t c = c0;
      for (auto &iv : wr[q][r]) {
        if (iv.first > c) break;
        if (iv.second > c) c = iv.second;
        if (c >= c1) return true;
      }
      return c >= c1;
    };
    for (size_t ti : finals) {
      const Task &t = tb.all[ti];
      for (int sq = 0; sq < t.nseg; ++sq) {
        const Seg &g = tb.segs[t.seg0 + sq];
        for (int side = 0; side < 2; ++side) {
          const View &v = tb.views[side == 0 ? g.a_map : g.b_map].first;
          for (int q = 0; q < 2; ++q) {
            if (v.addr < bufs[q] || v.addr >= bufs[q] + static_cast<uint64_t>(nrows[q] * rowb)) continue;
            const int64_t r0 = static_cast<int64_t>(v.addr - bufs[q]) / rowb;
            const int64_t c0 = side == 0 ? g.a_x : g.b_x;
            const int64_t c1 = c0 + (side == 0 ? t.rows : t.cols);
            for (int64_t r = r0; r < r0 + g.k_len; ++r)
              if (!covered(q, r, c0, c1)) {
                snprintf(buf, sizeof buf, "rect %zu: final product reads terminal row %lld not written", ri, (long long)r);
                return buf;
              }
          }
        }
      }
    }
  }
  // T coverage per rectangle: every T row Stage 3 reads has its columns [0, W_J)
  // written exactly once (by tiles of any width)
  for (size_t ri = 0; ri < tb.layouts.size(); ++ri) {
    if (tb.rect_triple[ri]) continue;
    const RectLayout &L = tb.layouts[ri];
    const bool left = tb.rect_left[ri] != 0;
    const LOp &X = left ? pc.XL : pc.XR;
    const uint64_t T = tb.rect_arena[ri] + static_cast<uint64_t>(L.Toffset);
    std::vector<std::vector<std::pair<int64_t, int64_t>>> wr(static_cast<size_t>(L.Trows));
    for (size_t ti = 0; ti < tb.all.size(); ++ti) {
      if (tb.task_rect[ti] != static_cast<int>(ri)) continue;
      const Task &t = tb.all[ti];
      const Out &o = tb.outs[t.out];
      if (o.kind == kOutC || reinterpret_cast<uint64_t>(o.ptr) != T) continue;
      auto add = [&](int64_t r0, int64_t n) {
        for (int64_t r = r0; r < r0 + n; ++r)
          if (r >= 0 && r < L.Trows) wr[r].push_back({t.col0, t.col0 + t.cols});
      };
      if (t.npiece == 0) add(t.row0, t.rows);
      for (int q = 0; q < t.npiece; ++q) add(tb.pieces[t.piece0 + q].dst0, tb.pieces[t.piece0 + q].len);
    }
    std::vector<uint8_t> needed(static_cast<size_t>(L.Trows), 0);
    for (int i = L.i0; i < L.i1; ++i)
      for (size_t pi = 0; pi < X.rowp[i].size(); ++pi)
        for (int64_t r = L.Toff[i][pi]; r < L.Toff[i][pi] + X.rowp[i][pi].v.cols; ++r) needed[r] = 1;
    for (int64_t r = 0; r < L.Trows; ++r) {
      auto &v = wr[r];
      std::sort(v.begin(), v.end());
      int64_t c = 0;
      for (auto &iv : v) {
        if (iv.first != c) {
          snprintf(buf, sizeof buf, "rect %zu: T row %lld written %s at column %lld", ri, (long long)r,
                   iv.first < c ? "twice" : "with a gap", (long long)c);
          return buf;
        }
        c = iv.second;
      }
      if (needed[r] && c != L.WJ) {
        snprintf(buf, sizeof buf, "rect %zu: T row %lld read by Stage 3 written up to column %lld of %lld", ri,
                 (long long)r, (long long)c, (long long)L.WJ);
        return buf;
      }
    }
  }
  return std::string();
}

cudaError_t record_start(tlr_handle_t h, int kind, std::pair<cudaEvent_t, cudaEvent_t> &ev) {
  if (!h->timing) return cudaSuccess;
  if (h->ev_free.empty()) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) return cudaErrorUnknown;
    h->ev_free.push_back({a, b});
  }
  ev = h->ev_free.back();
  h->ev_free.pop_back();
  h->ev_used.push_back({kind, ev});
  return cudaEventRecord(ev.first, h->stream);
}

cudaError_t record_stop(tlr_handle_t h, const std::pair<cudaEvent_t, cudaEvent_t> &ev) {
  if (!h->timing) return cudaSuccess;
  return cudaEventRecord(ev.second, h->stream);
}

}  // namespace

// ------------------------------------------------------------------ static scratch
// Device memory of tlr_gemm_static_scratch: one product's workspace, descriptor
// tables and counters. The CUDA runtime reserves it when it loads this
// translation unit's module (with lazy loading: at the first address lookup),
// never during a product.
static __device__ __align__(256) unsigned char g_static_scratch[TLR_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
struct StaticSlot {
  unsigned long long ctx_id = 0;   // context the address was looked up in (0: never)
  void *ptr = nullptr;
};
StaticSlot g_static_slot[kMaxDevices];

// Unique id of the calling thread's current context (cuCtxGetId ids are never
// reused within a process, unlike context handles); 0 when it cannot be read.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static bool looked = false;
  if (!looked) {
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
        qb == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
    looked = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_static_scratch on the current device. The lookup runs
// once per device and context: the first call on a device does it, and a call
// after that device's context was destroyed and re-created (cudaDeviceReset)
// does it again, so a stale address is never used. The host never takes the
// symbol itself as a device address.
tlr_status_t static_scratch_ptr(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return TLR_STATUS_CUDA_ERROR; }
  if (dev < 0 || dev >= kMaxDevices) return TLR_STATUS_UNSUPPORTED;
  const unsigned long long ctx = current_context_id();   // 0 until this thread has a current context
  std::lock_guard<std::mutex> lock(g_static_mu);
  StaticSlot &sl = g_static_slot[dev];
  if (!sl.ptr || ctx == 0 || sl.ctx_id != ctx) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return TLR_STATUS_CUDA_ERROR;
    }
    sl.ptr = ptr;
    sl.ctx_id = current_context_id();   // the lookup made the device's context current
  }
  *out = sl.ptr;
  return TLR_STATUS_OK;
}

}  // namespace

// ------------------------------------------------------------------ exported ABI
extern "C" {

const char *tlr_status_string(tlr_status_t s) {
  switch (s) {
    case TLR_STATUS_OK: return "TLR_STATUS_OK";
    case TLR_STATUS_INVALID_ARG: return "TLR_STATUS_INVALID_ARG";
    case TLR_STATUS_ALIGNMENT: return "TLR_STATUS_ALIGNMENT";
    case TLR_STATUS_WORKSPACE_TOO_SMALL: return "TLR_STATUS_WORKSPACE_TOO_SMALL";
    case TLR_STATUS_UNSUPPORTED: return "TLR_STATUS_UNSUPPORTED";
    case TLR_STATUS_CUDA_ERROR: return "TLR_STATUS_CUDA_ERROR";
    case TLR_STATUS_TIMEOUT: return "TLR_STATUS_TIMEOUT";
    case TLR_STATUS_NOT_INITIALIZED: return "TLR_STATUS_NOT_INITIALIZED";
  }
  return "TLR_STATUS_UNKNOWN";
}

tlr_status_t tlr_create(tlr_handle_t *handle, void *stream) {
  if (!handle) return TLR_STATUS_INVALID_ARG;
  *handle = nullptr;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) { cudaGetLastError(); return TLR_STATUS_NOT_INITIALIZED; }
  tlr_handle_s *h = new (std::nothrow) tlr_handle_s();
  if (!h) return TLR_STATUS_INVALID_ARG;
  h->stream = static_cast<cudaStream_t>(stream);
  if (cudaGetDevice(&h->device) != cudaSuccess) { cudaGetLastError(); delete h; return TLR_STATUS_NOT_INITIALIZED; }
  if (cudaMalloc(&h->d_err, 256) != cudaSuccess || cudaMemset(h->d_err, 0, 256) != cudaSuccess) {
    delete h;
    return TLR_STATUS_CUDA_ERROR;
  }
  *handle = h;
  return TLR_STATUS_OK;
}

tlr_status_t tlr_destroy(tlr_handle_t h) {
  if (!h) return TLR_STATUS_INVALID_ARG;
  cudaStreamSynchronize(h->stream);
  for (auto &e : h->ev_free) { cudaEventDestroy(e.first); cudaEventDestroy(e.second); }
  for (auto &e : h->ev_used) { cudaEventDestroy(e.second.first); cudaEventDestroy(e.second.second); }
  cudaFree(h->d_err);
  delete h;
  return TLR_STATUS_OK;
}

tlr_status_t tlr_set_stream(tlr_handle_t h, void *stream) {
  if (!h) return TLR_STATUS_INVALID_ARG;
  h->stream = static_cast<cudaStream_t>(stream);
  return TLR_STATUS_OK;
}

tlr_status_t tlr_analyze(tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A, const tlr_operand_t *B,
                         tlr_analysis_t *out) {
  if (!out || !A || !B) return TLR_STATUS_INVALID_ARG;
  if (A->kind != TLR_KIND_TLR || B->kind != TLR_KIND_TLR) return TLR_STATUS_UNSUPPORTED;
  PlanCore pc;
  tlr_status_t st = core_init(pc, opA, opB, A, B, false, 0);
  if (st) return st;
  const LOp &X = pc.XR, &Y = pc.YR;
  out->nt_i = X.nr; out->nt_k = X.nc; out->nt_j = Y.nc;
  int64_t W = 0, H = 0;
  for (int j = 0; j < Y.nc; ++j) W += Y.cd[j];
  for (int i = 0; i < X.nr; ++i) H += X.rd[i];
  int64_t sr = 0, sg = 0;
  for (int i = 0; i < X.nr; ++i) {
    int64_t rho = 0;
    for (int k = 0; k < X.nc; ++k) if (!X.dt(i, k)) rho += X.r(i, k);
    if (out->rho) out->rho[i] = rho;
    if (out->stage3_mnk) { out->stage3_mnk[3 * i] = X.rd[i]; out->stage3_mnk[3 * i + 1] = W; out->stage3_mnk[3 * i + 2] = rho; }
    sr += rho;
  }
  for (int j = 0; j < Y.nc; ++j) {
    int64_t g = 0;
    for (int k = 0; k < Y.nr; ++k) if (!Y.dt(k, j)) g += Y.r(k, j);
    if (out->gamma) out->gamma[j] = g;
    sg += g;
  }
  for (int k = 0; k < X.nc; ++k) {
    int64_t s = 0, G = 0;
    for (int i = 0; i < X.nr; ++i) if (!X.dt(i, k)) s += X.r(i, k);
    for (int j = 0; j < Y.nc; ++j) if (!Y.dt(k, j)) G += Y.r(k, j);
    if (out->sigma) out->sigma[k] = s;
    if (out->Gamma) out->Gamma[k] = G;
    if (out->stage1_mnk) { out->stage1_mnk[3 * k] = s; out->stage1_mnk[3 * k + 1] = G; out->stage1_mnk[3 * k + 2] = X.cd[k]; }
  }
  out->F_R = final_cost(X, 0, X.nr, W);
  out->F_L = final_cost(pc.XL, 0, pc.XL.nr, H);
  out->F_P = triple_cost(pc);
  out->order = out->F_L < out->F_R ? TLR_ORDER_LEFT : TLR_ORDER_RIGHT;
  out->T_right_rows = sr; out->T_right_cols = W;
  out->T_left_rows = H; out->T_left_cols = sg;
  int64_t prods = 0;
  std::set<std::pair<int32_t, int32_t>> shapes;
  for (int i = 0; i < X.nr; ++i)
    for (int k = 0; k < X.nc; ++k)
      for (int j = 0; j < Y.nc; ++j) {
        if (X.dt(i, k) || Y.dt(k, j)) continue;
        if (X.r(i, k) <= 0 || Y.r(k, j) <= 0) continue;
        ++prods;
        shapes.insert({X.r(i, k), Y.r(k, j)});
      }
  out->coupling_products = prods;
  out->distinct_shapes = static_cast<int64_t>(shapes.size());
  return TLR_STATUS_OK;
}

tlr_status_t tlr_gemm_workspace_bytes(tlr_handle_t h, tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A,
                                      const tlr_operand_t *B, int runs, size_t *bytes) {
  return tlr_gemm_workspace_bytes_for_order(h, opA, opB, A, B, runs, TLR_ORDER_AUTO, bytes);
}

tlr_status_t tlr_gemm_workspace_bytes_for_order(tlr_handle_t h, tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A,
                                                const tlr_operand_t *B, int runs, tlr_order_t order, size_t *bytes) {
  (void)h;
  if (!bytes) return TLR_STATUS_INVALID_ARG;
  if (order < TLR_ORDER_AUTO || order > TLR_ORDER_PER_RECT) return TLR_STATUS_INVALID_ARG;
  PlanCore pc;
  tlr_status_t st = core_init(pc, opA, opB, A, B, false, 0);
  if (st) return st;
  const int es = elem_size(pc.pv.dtype);
  if (runs <= 0) runs = 1;
  std::vector<Rect> rects;
  int na = 1;
  int64_t whole = 0;   // the largest one-rectangle workspace of any order the plan may take
  if (pc.can_right) whole = std::max(whole, rect_bytes(pc, 0, pc.nI, 0, pc.nJ, false, es));
  if (pc.can_left) whole = std::max(whole, rect_bytes(pc, 0, pc.nI, 0, pc.nJ, true, es));
  if (can_triple(pc)) whole = std::max(whole, rect_bytes_triple(pc, 0, pc.nI, 0, pc.nJ, es));
  int64_t hi = pc.fixed + 2 * whole;
  if (order == TLR_ORDER_TRIPLE && !can_triple(pc)) return TLR_STATUS_UNSUPPORTED;
  if (!plan_split(pc, hi, order, es, rects, na)) return TLR_STATUS_INVALID_ARG;
  const int min_runs = static_cast<int>(rects.size());
  runs = std::max(runs, min_runs);
  int64_t lo = pc.fixed;
  // smallest budget whose plan has at most `runs` rectangles
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (plan_split(pc, mid, order, es, rects, na) && static_cast<int>(rects.size()) <= runs) hi = mid;
    else lo = mid + 1;
  }
  plan_split(pc, hi, order, es, rects, na);
  *bytes = static_cast<size_t>(pc.fixed + na * align_up(max_rect_bytes(pc, rects, es), 256));
  return TLR_STATUS_OK;
}

// Buffers the kernels read or write through TMA must be device memory
// (cudaMalloc or managed); a host pointer, pinned or not, is refused before any
// table is built or kernel launched.
bool device_memory(const void *ptr) {
  if (!ptr) return true;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

bool operand_on_device(const tlr_operand_t *X) {
  if (X->kind == TLR_KIND_DENSE) return device_memory(X->data);
  for (const void *q : {X->U, X->V, X->D, X->bu_U, X->bu_V, X->bv_U, X->bv_V, X->gamma})
    if (!device_memory(q)) return false;
  return true;
}

tlr_status_t tlr_plan_create(tlr_handle_t h, tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A,
                             const tlr_operand_t *B, void *workspace, size_t workspace_bytes,
                             tlr_order_t order, tlr_plan_t *plan_out) {
  if (!h || !plan_out) return TLR_STATUS_INVALID_ARG;
  *plan_out = nullptr;
  if (order < TLR_ORDER_AUTO || order > TLR_ORDER_PER_RECT) return TLR_STATUS_INVALID_ARG;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return TLR_STATUS_ALIGNMENT;
  const uint64_t ws = reinterpret_cast<uint64_t>(workspace);
  PlanCore pc;
  tlr_status_t st = core_init(pc, opA, opB, A, B, true, ws ? ws : 256);
  if (st) return st;
  if (!operand_on_device(A) || !operand_on_device(B) || !device_memory(workspace)) return TLR_STATUS_INVALID_ARG;
  const int es = elem_size(pc.pv.dtype);
  const bool tf32 = pc.pv.dtype == TLR_F32;
  std::vector<Rect> rects;
  int narenas = 1;
  if (order == TLR_ORDER_TRIPLE && !can_triple(pc)) return TLR_STATUS_UNSUPPORTED;
  if (!plan_split(pc, static_cast<int64_t>(workspace_bytes), order, es, rects, narenas))
    return TLR_STATUS_WORKSPACE_TOO_SMALL;
  const int64_t need = pc.fixed + narenas * align_up(max_rect_bytes(pc, rects, es), 256);
  if (need > 0 && !workspace) return TLR_STATUS_INVALID_ARG;

  tlr_plan_s *p = new (std::nothrow) tlr_plan_s();
  if (!p) return TLR_STATUS_INVALID_ARG;
  p->h = h;
  p->tf32 = tf32;
  p->f16 = pc.pv.dtype == TLR_F16;
  p->Cm = pc.pv.Cm;
  p->Cn = pc.pv.Cn;
  p->round_src = pc.round_src;
  p->round_dst = pc.round_dst;
  p->round_n = pc.round_n;
  p->bn = choose_bn(pc);

  Tables tb;
  tb.bn = p->bn;
  tb.pair = p->pair = choose_pair(pc, p->bn);
  tb.prep_pair = choose_prep_pair(pc, p->bn, tb.pair);
  tb.l1_pair = choose_l1_pair(pc, tb.prep_pair, tb.pair);
  choose_prep_widths(tb);
  st = build_tables(pc, rects, narenas, ws, false, tb);
  if (st) { delete p; return st; }
  p->launches = tb.launches;
  p->rects = abi_rects(rects);
  p->info = tb.info;
  tlr_plan_info_t &info = p->info;
  info.workspace_bytes = static_cast<size_t>(need);
  info.launches = static_cast<int64_t>(p->launches.size()) + (p->round_n.empty() ? 0 : 1);
  if (static_cast<size_t>(need) > workspace_bytes) { delete p; return TLR_STATUS_WORKSPACE_TOO_SMALL; }
  std::vector<CUtensorMap> &maps = tb.maps;
  std::vector<Task> &all = tb.all;
  std::vector<Seg> &segs = tb.segs;
  std::vector<Piece> &pieces = tb.pieces;
  std::vector<Out> &outs = tb.outs;

  // one device allocation for all tables: maps first (64-byte aligned)
  const size_t szm = maps.size() * sizeof(CUtensorMap);
  const size_t szt = align_up(static_cast<int64_t>(all.size() * sizeof(Task)), 256);
  const size_t szs = align_up(static_cast<int64_t>(segs.size() * sizeof(Seg)), 256);
  const size_t szp = align_up(static_cast<int64_t>(pieces.size() * sizeof(Piece)), 256);
  const size_t szo = align_up(static_cast<int64_t>(outs.size() * sizeof(Out)), 256);
  std::vector<TJob> tj;
  int64_t tiles = 0;
  for (const TJobHost &j : pc.tjobs) {
    TJob d;
    memset(&d, 0, sizeof d);
    d.src = reinterpret_cast<const float *>(j.src);
    d.dst = reinterpret_cast<float *>(j.dst);
    d.src_ld = j.src_ld; d.dst_ld = j.dst_ld; d.rows = j.rows; d.cols = j.cols; d.tile0 = tiles;
    tiles += ceil_div(j.rows, 32) * ceil_div(j.cols, 32);
    tj.push_back(d);
  }
  const size_t szj = align_up(static_cast<int64_t>(tj.size() * sizeof(TJob)), 256);
  const size_t szc = align_up(static_cast<int64_t>((tb.launches.size() + tb.counter_counts.size()) * sizeof(unsigned int)), 256);
  const size_t om = 0, ot = align_up(static_cast<int64_t>(szm), 256), os = ot + szt, op = os + szs, oo = op + szp;
  const size_t oj = oo + szo, oc = oj + szj;
  const size_t total = oc + szc + 256;
  std::vector<uint8_t> host(total, 0);
  if (szm) memcpy(host.data() + om, maps.data(), szm);
  if (!all.empty()) memcpy(host.data() + ot, all.data(), all.size() * sizeof(Task));
  if (!segs.empty()) memcpy(host.data() + os, segs.data(), segs.size() * sizeof(Seg));
  if (!pieces.empty()) memcpy(host.data() + op, pieces.data(), pieces.size() * sizeof(Piece));
  if (!outs.empty()) memcpy(host.data() + oo, outs.data(), outs.size() * sizeof(Out));
  if (!tj.empty()) memcpy(host.data() + oj, tj.data(), tj.size() * sizeof(TJob));
  if (cudaMallocAsync(&p->d_tables, total, h->stream) != cudaSuccess) { cudaGetLastError(); delete p; return TLR_STATUS_CUDA_ERROR; }
  if (cudaMemcpyAsync(p->d_tables, host.data(), total, cudaMemcpyHostToDevice, h->stream) != cudaSuccess ||
      cudaStreamSynchronize(h->stream) != cudaSuccess) {
    cudaFreeAsync(p->d_tables, h->stream);
    delete p;
    return TLR_STATUS_CUDA_ERROR;
  }
  uint8_t *dt = static_cast<uint8_t *>(p->d_tables);
  p->d_maps = dt + om;
  p->d_tasks = reinterpret_cast<const Task *>(dt + ot);
  p->d_segs = reinterpret_cast<const Seg *>(dt + os);
  p->d_pieces = reinterpret_cast<const Piece *>(dt + op);
  p->d_outs = reinterpret_cast<const Out *>(dt + oo);
  p->d_tjobs = reinterpret_cast<const TJob *>(dt + oj);
  p->d_counters = reinterpret_cast<unsigned int *>(dt + oc);
  p->counters_bytes = szc;
  p->ntjobs = static_cast<int>(tj.size());
  p->ttiles = tiles;
  *plan_out = p;
  return TLR_STATUS_OK;
}

tlr_status_t tlr_debug_check_plan(tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A, const tlr_operand_t *B,
                                  size_t workspace_bytes, tlr_order_t order, tlr_plan_info_t *info,
                                  char *msg, size_t msg_len) {
  if (msg && msg_len) msg[0] = 0;
  if (order < TLR_ORDER_AUTO || order > TLR_ORDER_PER_RECT) return TLR_STATUS_INVALID_ARG;
  const uint64_t ws = 0x100000000000ull;   // a stand-in address: nothing is dereferenced
  PlanCore pc;
  tlr_status_t st = core_init(pc, opA, opB, A, B, true, ws);
  if (st) return st;
  const int es = elem_size(pc.pv.dtype);
  std::vector<Rect> rects;
  int narenas = 1;
  if (order == TLR_ORDER_TRIPLE && !can_triple(pc)) return TLR_STATUS_UNSUPPORTED;
  if (!plan_split(pc, static_cast<int64_t>(workspace_bytes), order, es, rects, narenas))
    return TLR_STATUS_WORKSPACE_TOO_SMALL;
  Tables tb;
  tb.bn = choose_bn(pc);
  tb.pair = choose_pair(pc, tb.bn);
  tb.prep_pair = choose_prep_pair(pc, tb.bn, tb.pair);
  tb.l1_pair = choose_l1_pair(pc, tb.prep_pair, tb.pair);
  choose_prep_widths(tb);
  st = build_tables(pc, rects, narenas, ws, true, tb);
  if (st) return st;
  const int64_t need = pc.fixed + narenas * align_up(max_rect_bytes(pc, rects, es), 256);
  tb.info.workspace_bytes = static_cast<size_t>(need);
  tb.info.launches = static_cast<int64_t>(tb.launches.size());
  if (info) *info = tb.info;
  const std::string why = validate_tables(pc, tb, ws, std::max<int64_t>(need, static_cast<int64_t>(workspace_bytes)));
  if (!why.empty()) {
    if (msg && msg_len) { strncpy(msg, why.c_str(), msg_len - 1); msg[msg_len - 1] = 0; }
    return TLR_STATUS_INVALID_ARG;
  }
  return TLR_STATUS_OK;
}

tlr_status_t tlr_plan_info(tlr_plan_t plan, tlr_plan_info_t *info) {
  if (!plan || !info) return TLR_STATUS_INVALID_ARG;
  *info = plan->info;
  return TLR_STATUS_OK;
}

tlr_status_t tlr_plan_rects(tlr_plan_t plan, tlr_rect_t *rects, int32_t capacity, int32_t *count) {
  if (!plan) return TLR_STATUS_INVALID_ARG;
  return copy_rects(plan->rects, rects, capacity, count);
}

tlr_status_t tlr_debug_plan_rects(tlr_op_t opA, tlr_op_t opB, const tlr_operand_t *A, const tlr_operand_t *B,
                                  size_t workspace_bytes, tlr_order_t order, tlr_rect_t *rects, int32_t capacity,
                                  int32_t *count) {
  if (order < TLR_ORDER_AUTO || order > TLR_ORDER_PER_RECT) return TLR_STATUS_INVALID_ARG;
  PlanCore pc;
  tlr_status_t st = core_init(pc, opA, opB, A, B, false, 0x100000000000ull);
  if (st) return st;
  std::vector<Rect> rs;
  int narenas = 1;
  if (order == TLR_ORDER_TRIPLE && !can_triple(pc)) return TLR_STATUS_UNSUPPORTED;
  if (!plan_split(pc, static_cast<int64_t>(workspace_bytes), order, elem_size(pc.pv.dtype), rs, narenas))
    return TLR_STATUS_WORKSPACE_TOO_SMALL;
  return copy_rects(abi_rects(rs), rects, capacity, count);
}

// Tensor maps of C for the epilogue's bulk stores (see Params::cmap). A map
// that cannot be encoded only disables the bulk stores.
bool encode_c_maps(Params &prm, float *C, int64_t ldc, int64_t m, int64_t n) {
  auto fn = encode_fn();
  if (!fn || m <= 0 || n <= 0) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(m), static_cast<cuuint64_t>(n)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc) * 4u};
  cuuint32_t estr[2] = {1, 1};
  const cuuint32_t boxes[2][2] = {{32, 16}, {16, 32}};
  const CUtensorMapSwizzle sw[2] = {CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_SWIZZLE_64B};
  for (int q = 0; q < 2; ++q) {
    CUresult r = fn(&prm.cmap[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, strides, boxes[q], estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw[q], CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  return true;
}

tlr_status_t tlr_plan_execute(tlr_plan_t p, float alpha, float beta, float *C, int64_t ldc) {
  if (!p || !C) return TLR_STATUS_INVALID_ARG;
  if (ldc < p->Cm || (ldc % 4)) return ldc < p->Cm ? TLR_STATUS_INVALID_ARG : TLR_STATUS_ALIGNMENT;
  if (!aligned16(C)) return TLR_STATUS_ALIGNMENT;
  if (!device_memory(C)) return TLR_STATUS_INVALID_ARG;
  tlr_handle_t h = p->h;
  const int sms = device_sms();
  std::pair<cudaEvent_t, cudaEvent_t> ev;
  if (alpha == 0.f) {
    if (record_start(h, kKindScale, ev) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
    cudaError_t e = launch_scale_c(C, ldc, p->Cm, p->Cn, beta, 4 * sms, h->stream);
    if (e != cudaSuccess || record_stop(h, ev) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
    return TLR_STATUS_OK;
  }
  if (!p->round_n.empty()) {
    if (record_start(h, kKindRound, ev) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
    cudaError_t e = launch_round_tf32(p->round_src.data(), p->round_dst.data(), p->round_n.data(),
                                      static_cast<int>(p->round_n.size()), 4 * sms, h->stream);
    if (e == cudaSuccess)
      e = launch_transpose_round(p->d_tjobs, p->ntjobs, p->ttiles,
                                 static_cast<int>(std::min<int64_t>(p->ttiles, 16 * sms)), h->stream);
    if (e != cudaSuccess || record_stop(h, ev) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  }
  Params prm;
  memset(&prm, 0, sizeof prm);
  prm.maps = p->d_maps;
  prm.segs = p->d_segs;
  prm.pieces = p->d_pieces;
  prm.outs = p->d_outs;
  prm.C = C;
  prm.ldc = ldc;
  prm.alpha = alpha;
  prm.beta = beta;
  prm.bn = p->bn;
  prm.err = h->d_err;
  prm.wait_limit_ns = h->wait_limit_ns;
  prm.cmap_ok = encode_c_maps(prm, C, ldc, p->Cm, p->Cn) ? 1 : 0;
  prm.f16 = p->f16 ? 1 : 0;
  // one ticket per launch, then the dependency counters; all start at zero
  prm.counters = p->d_counters + p->launches.size();
  if (cudaMemsetAsync(p->d_counters, 0, p->counters_bytes, h->stream) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  for (size_t li = 0; li < p->launches.size(); ++li) {
    const Launch &l = p->launches[li];
    prm.ticket = p->d_counters + li;
    prm.bn = l.bn > 0 ? l.bn : p->bn;
    prm.tasks = p->d_tasks + l.t0;
    prm.ntasks = static_cast<int32_t>(l.t1 - l.t0);
    int grid = static_cast<int>(std::min<int64_t>(sms, l.t1 - l.t0));
    if (l.pair == 2) {
      const int pairs = max_resident_pairs(p->tf32);
      if (pairs <= 0) return TLR_STATUS_UNSUPPORTED;
      grid = 2 * static_cast<int>(std::min<int64_t>(pairs, l.t1 - l.t0));
    } else if (l.pair == 4) {   // clusters of two pairs, one group of 2 kTicketBatch tickets each at a time
      const int quads = max_resident_quads(p->tf32);
      if (quads <= 0) return TLR_STATUS_UNSUPPORTED;
      grid = 4 * static_cast<int>(std::min<int64_t>(quads, (l.t1 - l.t0) / (2 * kTicketBatch)));
    }
    if (record_start(h, l.kind, ev) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
    if (launch_task_gemm(p->tf32, l.pair, prm, grid, h->stream) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
    if (record_stop(h, ev) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  }
  return TLR_STATUS_OK;
}

tlr_status_t tlr_plan_destroy(tlr_plan_t p) {
  if (!p) return TLR_STATUS_INVALID_ARG;
  if (p->d_tables) cudaFreeAsync(p->d_tables, p->h->stream);
  delete p;
  return TLR_STATUS_OK;
}

tlr_status_t tlr_gemm(tlr_handle_t h, tlr_op_t opA, tlr_op_t opB, float alpha, const tlr_operand_t *A,
                      const tlr_operand_t *B, float beta, float *C, int64_t ldc, void *workspace,
                      size_t workspace_bytes) {
  tlr_plan_t p = nullptr;
  tlr_status_t st = tlr_plan_create(h, opA, opB, A, B, workspace, workspace_bytes, TLR_ORDER_AUTO, &p);
  if (st) return st;
  st = tlr_plan_execute(p, alpha, beta, C, ldc);
  tlr_plan_destroy(p);
  return st;
}

// For callers that may not allocate device memory while they run a product:
// code whose allocator owns every free byte of the device, or loops that must
// not touch the allocator (allocation can synchronise the device and take
// milliseconds). Workspace, tables and counters of the product go into
// g_static_scratch; the tables are uploaded from host memory with one
// stream-ordered copy. Nothing is allocated or freed on the device.
tlr_status_t tlr_gemm_static_scratch(tlr_handle_t h, tlr_op_t opA, tlr_op_t opB, float alpha,
                                     const tlr_operand_t *A, const tlr_operand_t *B, float beta, float *C,
                                     int64_t ldc) {
  if (!h || !C) return TLR_STATUS_INVALID_ARG;
  if (!aligned16(C) || ldc % 4) return TLR_STATUS_ALIGNMENT;
  {
    // the scratch address is per device: the current one must be the handle's
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return TLR_STATUS_CUDA_ERROR; }
    if (dev != h->device) return TLR_STATUS_INVALID_ARG;
  }
  void *scratch = nullptr;
  tlr_status_t st = static_scratch_ptr(&scratch);
  if (st) return st;
  const uint64_t ws = reinterpret_cast<uint64_t>(scratch);   // the workspace comes first
  PlanCore pc;
  st = core_init(pc, opA, opB, A, B, true, ws);
  if (st) return st;
  if (ldc < pc.pv.Cm) return TLR_STATUS_INVALID_ARG;
  if (!operand_on_device(A) || !operand_on_device(B) || !device_memory(C)) return TLR_STATUS_INVALID_ARG;
  const int es = elem_size(pc.pv.dtype);
  std::vector<Rect> rects;
  int narenas = 1;
  constexpr int64_t kTableReserve = 2 << 20;   // the tables of any product that fits take far less
  if (!plan_split(pc, static_cast<int64_t>(TLR_STATIC_SCRATCH_BYTES) - kTableReserve, TLR_ORDER_AUTO, es, rects, narenas))
    return TLR_STATUS_WORKSPACE_TOO_SMALL;
  const int64_t need = pc.fixed + narenas * align_up(max_rect_bytes(pc, rects, es), 256);

  tlr_plan_s p;
  p.h = h;
  p.tf32 = pc.pv.dtype == TLR_F32;
  p.f16 = pc.pv.dtype == TLR_F16;
  p.Cm = pc.pv.Cm;
  p.Cn = pc.pv.Cn;
  p.round_src = pc.round_src;
  p.round_dst = pc.round_dst;
  p.round_n = pc.round_n;
  p.bn = choose_bn(pc);
  Tables tb;
  tb.bn = p.bn;
  tb.pair = p.pair = choose_pair(pc, p.bn);
  tb.prep_pair = choose_prep_pair(pc, p.bn, tb.pair);
  tb.l1_pair = choose_l1_pair(pc, tb.prep_pair, tb.pair);
  choose_prep_widths(tb);
  st = build_tables(pc, rects, narenas, ws, false, tb);
  if (st) return st;
  p.launches = tb.launches;
  p.info = tb.info;

  // tables after the workspace: tensor maps, tasks, segments, pieces, outputs,
  // transpose jobs, then the counters (one ticket per launch, then the
  // dependency counters), which tlr_plan_execute zeroes on the stream
  std::vector<TJob> tj;
  int64_t tiles = 0;
  for (const TJobHost &j : pc.tjobs) {
    TJob d;
    memset(&d, 0, sizeof d);
    d.src = reinterpret_cast<const float *>(j.src);
    d.dst = reinterpret_cast<float *>(j.dst);
    d.src_ld = j.src_ld; d.dst_ld = j.dst_ld; d.rows = j.rows; d.cols = j.cols; d.tile0 = tiles;
    tiles += ceil_div(j.rows, 32) * ceil_div(j.cols, 32);
    tj.push_back(d);
  }
  auto bytes_of = [](size_t n, size_t sz) { return static_cast<size_t>(align_up(static_cast<int64_t>(n * sz), 256)); };
  const size_t ot = bytes_of(tb.maps.size(), sizeof(CUtensorMap));
  const size_t os = ot + bytes_of(tb.all.size(), sizeof(Task));
  const size_t op = os + bytes_of(tb.segs.size(), sizeof(Seg));
  const size_t oo = op + bytes_of(tb.pieces.size(), sizeof(Piece));
  const size_t oj = oo + bytes_of(tb.outs.size(), sizeof(Out));
  const size_t oc = oj + bytes_of(tj.size(), sizeof(TJob));
  const size_t szc = bytes_of(tb.launches.size() + tb.counter_counts.size(), sizeof(unsigned int));
  const size_t total = oc + szc;
  const size_t t0 = static_cast<size_t>(align_up(need, 256));
  if (t0 + total > static_cast<size_t>(TLR_STATIC_SCRATCH_BYTES)) return TLR_STATUS_WORKSPACE_TOO_SMALL;
  std::vector<uint8_t> host(oc, 0);
  if (!tb.maps.empty()) memcpy(host.data(), tb.maps.data(), tb.maps.size() * sizeof(CUtensorMap));
  if (!tb.all.empty()) memcpy(host.data() + ot, tb.all.data(), tb.all.size() * sizeof(Task));
  if (!tb.segs.empty()) memcpy(host.data() + os, tb.segs.data(), tb.segs.size() * sizeof(Seg));
  if (!tb.pieces.empty()) memcpy(host.data() + op, tb.pieces.data(), tb.pieces.size() * sizeof(Piece));
  if (!tb.outs.empty()) memcpy(host.data() + oo, tb.outs.data(), tb.outs.size() * sizeof(Out));
  if (!tj.empty()) memcpy(host.data() + oj, tj.data(), tj.size() * sizeof(TJob));
  uint8_t *dt = static_cast<uint8_t *>(scratch) + t0;
  // From pageable memory the copy returns once `host` has been staged, so it
  // may go out of scope; the copy stays ordered after earlier work on the stream.
  if (oc && cudaMemcpyAsync(dt, host.data(), oc, cudaMemcpyHostToDevice, h->stream) != cudaSuccess) {
    cudaGetLastError();
    return TLR_STATUS_CUDA_ERROR;
  }
  p.d_maps = dt;
  p.d_tasks = reinterpret_cast<const Task *>(dt + ot);
  p.d_segs = reinterpret_cast<const Seg *>(dt + os);
  p.d_pieces = reinterpret_cast<const Piece *>(dt + op);
  p.d_outs = reinterpret_cast<const Out *>(dt + oo);
  p.d_tjobs = reinterpret_cast<const TJob *>(dt + oj);
  p.d_counters = reinterpret_cast<unsigned int *>(dt + oc);
  p.counters_bytes = szc;
  p.ntjobs = static_cast<int>(tj.size());
  p.ttiles = tiles;
  return tlr_plan_execute(&p, alpha, beta, C, ldc);
}

tlr_status_t tlr_get_device_status(tlr_handle_t h) {
  if (!h) return TLR_STATUS_INVALID_ARG;
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  unsigned int err = 0;
  if (cudaMemcpy(&err, h->d_err, sizeof err, cudaMemcpyDeviceToHost) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  if (err) {
    cudaMemset(h->d_err, 0, sizeof err);
    return TLR_STATUS_TIMEOUT;
  }
  return TLR_STATUS_OK;
}

tlr_status_t tlr_set_timing(tlr_handle_t h, int enabled) {
  if (!h) return TLR_STATUS_INVALID_ARG;
  h->timing = enabled != 0;
  return TLR_STATUS_OK;
}

static tlr_status_t collect_timing(tlr_handle_t h) {
  if (h->ev_used.empty()) return TLR_STATUS_OK;
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  for (auto &u : h->ev_used) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, u.second.first, u.second.second) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
    h->ms[u.first] += ms;
    h->count[u.first] += 1;
    h->ev_free.push_back(u.second);
  }
  h->ev_used.clear();
  return TLR_STATUS_OK;
}

tlr_status_t tlr_get_timing(tlr_handle_t h, int kind, double *ms, int64_t *launches) {
  if (!h || kind < 0 || kind >= kNumKinds) return TLR_STATUS_INVALID_ARG;
  tlr_status_t st = collect_timing(h);
  if (st) return st;
  if (ms) *ms = h->ms[kind];
  if (launches) *launches = h->count[kind];
  return TLR_STATUS_OK;
}

tlr_status_t tlr_reset_timing(tlr_handle_t h) {
  if (!h) return TLR_STATUS_INVALID_ARG;
  tlr_status_t st = collect_timing(h);
  for (int k = 0; k < kNumKinds; ++k) { h->ms[k] = 0; h->count[k] = 0; }
  return st;
}

tlr_status_t tlr_set_wait_limit_us(tlr_handle_t h, int64_t limit_us) {
  if (!h || limit_us <= 0) return TLR_STATUS_INVALID_ARG;
  h->wait_limit_ns = static_cast<unsigned long long>(limit_us) * 1000ull;
  return TLR_STATUS_OK;
}

tlr_status_t tlr_debug_unsatisfied_wait(tlr_handle_t h) {
  if (!h) return TLR_STATUS_INVALID_ARG;
  Params prm;
  memset(&prm, 0, sizeof prm);
  prm.err = h->d_err;
  prm.wait_limit_ns = h->wait_limit_ns;
  if (launch_unsatisfied_wait(prm, h->stream) != cudaSuccess) return TLR_STATUS_CUDA_ERROR;
  return TLR_STATUS_OK;
}

}  // extern "C"

// Handle access for the library's other translation unit (tlr_compress.cu).
namespace tlr {
cudaStream_t handle_stream(tlr_handle_t h) { return h->stream; }
bool handle_on_current_device(tlr_handle_t h) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return false; }
  return dev == h->device;
}
bool is_device_pointer(const void *p) { return p != nullptr && device_memory(p); }
}  // namespace tlr
