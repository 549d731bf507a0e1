/*
 * CPU fp64 oracle for the Tile-Low-Rank GEMM   C <- alpha * op(A) * op(B) + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the package smoke check and the
 * benchmark's CPU-baseline leg are the only callers. It shares no code, header,
 * table or helper with the GPU path, and the GPU path never calls it.
 *
 * What it computes is the plain definition of the product ("Tile-Low-Rank GEMM:
 * Designing Storage Around the Contraction", opening section: dense C, one or
 * both operands in TLR format). Each TLR operand is expanded into the dense
 * matrix it stands for, tile by tile:
 *   - off-diagonal tile (i,k) is U_ik V_ik^T with its own rank r_ik
 *     (same page, section "Many small GEMMs");
 *   - diagonal tiles are dense; the boundary column u, boundary row v^T and the
 *     dense corner gamma cover N not a multiple of b
 *     ("TLR Matrix Multiplication", section "Introduction: TLR GEMM");
 *   - op(X) = X^T swaps the roles of the factor families
 *     (first page, section "Where fusion stops", paragraph "Transposes"),
 *     which the expansion realises simply by reading column r of X for row r
 *     of X^T.
 * Every requested output entry is then alpha * sum_t opA[r,t] * opB[t,c]
 * (+ beta * C[r,c]) summed in fp64 over the contraction index t in ascending
 * order, i.e. over contraction tiles k in ascending order. When beta == 0, C is
 * not read; when alpha == 0 the operands are not read (BLAS convention).
 *
 * Storage read here (the format of the pages, with the readings of ambiguous
 * points stated once): outer factors U packed by tile row, inner factors V
 * packed by tile column, each factor column-major with leading dimension equal
 * to its own dense dimension and exactly r_ik columns; dense tiles skipped in
 * the packing; the boundary column's factors in bu_U/bu_V (ascending i), the
 * boundary row's in bv_U/bv_V (ascending j), the corner in gamma. Offsets are
 * recomputed here from the rank array with this file's own code.
 *
 * Build: cc -O2 -fopenmp -shared -fPIC tlr_oracle.c -o libtlr_oracle.so
 */
#include <math.h>
#include <stdint.h>
/* ORC_MUTATE plants a known mistake (tests check that the pins catch it):
 * 1 drops the dense diagonal tiles, 2 reads V with the tile-row packing order,
 * 3 uses V_ik[c, t] as V_ik[t, c] (transposed factor), 4 flips the sign of beta. */
#ifndef ORC_MUTATE
#define ORC_MUTATE 0
#endif
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t kind;        /* 0 = TLR, 1 = dense */
    int32_t diag_dense;  /* TLR: diagonal tiles stored dense */
    int64_t rows, cols;  /* dense dimensions of the stored matrix (before op) */
    int64_t b;           /* nominal tile size (TLR) */
    const int32_t *ranks;/* TLR: nt_r x nt_c, row-major; dense tiles ignored */
    const float *U, *V, *D;
    const float *bu_U, *bu_V, *bv_U, *bv_V, *gamma;
    const float *dense;  /* dense: column-major values */
    int64_t ld;          /* dense: leading dimension */
} orc_mat;

enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_BAD_RANK = 2, ORC_NO_MEMORY = 3 };

/* ----------------------------------------------------------- tile geometry */
typedef struct {
    const orc_mat *X;
    int64_t ntr, ntc;     /* tile grid */
    int64_t m;            /* interior tile count per axis when there is a boundary */
    int64_t brem;         /* boundary tile size (0: none) */
    int64_t *ucol, *vcol; /* packed column index of each interior low-rank tile */
} orc_geo;

static int64_t ntiles(int64_t n, int64_t b) { return (n + b - 1) / b; }

static int64_t tdim(const orc_geo *g, int64_t t, int64_t n) {
    int64_t b = g->X->b;
    int64_t d = n - t * b;
    return d < b ? d : b;
}

static int is_dense_tile(const orc_geo *g, int64_t i, int64_t k) {
    return g->X->diag_dense && i == k;
}

static int64_t rank_of(const orc_geo *g, int64_t i, int64_t k) {
    if (is_dense_tile(g, i, k)) return 0;
    return g->X->ranks[i * g->ntc + k];
}

static int geo_init(orc_geo *g, const orc_mat *X) {
    memset(g, 0, sizeof(*g));
    g->X = X;
    if (X->kind != 0) return ORC_OK;
    if (X->b <= 0 || X->rows <= 0 || X->cols <= 0 || !X->ranks) return ORC_BAD_ARG;
    g->ntr = ntiles(X->rows, X->b);
    g->ntc = ntiles(X->cols, X->b);
    int boundary = (X->rows % X->b) != 0 || (X->cols % X->b) != 0;
    if (boundary) {
        if (!X->diag_dense || X->rows != X->cols) return ORC_BAD_ARG;
        g->m = X->rows / X->b;
        g->brem = X->rows - g->m * X->b;
    } else {
        g->m = -1;
        g->brem = 0;
    }
    if (X->diag_dense && X->rows != X->cols) return ORC_BAD_ARG;
    for (int64_t i = 0; i < g->ntr; i++)
        for (int64_t k = 0; k < g->ntc; k++) {
            int64_t r = rank_of(g, i, k);
            int64_t di = tdim(g, i, X->rows), dk = tdim(g, k, X->cols);
            if (r < 0 || r > di || r > dk) return ORC_BAD_RANK;
        }
    int64_t nr = boundary ? g->m : g->ntr;   /* interior rows / cols */
    int64_t nc = boundary ? g->m : g->ntc;
    g->ucol = (int64_t *)calloc((size_t)(g->ntr * g->ntc), sizeof(int64_t));
    g->vcol = (int64_t *)calloc((size_t)(g->ntr * g->ntc), sizeof(int64_t));
    if (!g->ucol || !g->vcol) return ORC_NO_MEMORY;
    /* U: tile rows ascending, then tile columns ascending */
    int64_t c = 0;
    for (int64_t i = 0; i < nr; i++)
        for (int64_t k = 0; k < nc; k++) {
            if (is_dense_tile(g, i, k)) continue;
            g->ucol[i * g->ntc + k] = c;
            c += rank_of(g, i, k);
        }
    /* V: tile columns ascending, then tile rows ascending */
    c = 0;
    for (int64_t k = 0; k < nc; k++)
        for (int64_t i = 0; i < nr; i++) {
            if (is_dense_tile(g, i, k)) continue;
            g->vcol[i * g->ntc + k] = c;
            c += rank_of(g, i, k);
        }
    if (boundary) {
        int64_t m = g->m;
        c = 0;  /* boundary column: tiles (i, m), ascending i */
        for (int64_t i = 0; i < m; i++) { g->ucol[i * g->ntc + m] = c; g->vcol[i * g->ntc + m] = c; c += rank_of(g, i, m); }
        c = 0;  /* boundary row: tiles (m, j), ascending j */
        for (int64_t j = 0; j < m; j++) { g->ucol[m * g->ntc + j] = c; g->vcol[m * g->ntc + j] = c; c += rank_of(g, m, j); }
    }
    return ORC_OK;
}

static void geo_free(orc_geo *g) {
    free(g->ucol);
    free(g->vcol);
}

/* Pointers to the factors of low-rank tile (i,k): U_ik is d_i x r (ld d_i),
 * V_ik is d_k x r (ld d_k). */
static void tile_factors(const orc_geo *g, int64_t i, int64_t k, const float **Up, const float **Vp) {
    const orc_mat *X = g->X;
    int64_t di = tdim(g, i, X->rows), dk = tdim(g, k, X->cols);
    int64_t uc = g->ucol[i * g->ntc + k], vc = g->vcol[i * g->ntc + k];
    if (ORC_MUTATE == 2) vc = uc;
    if (g->brem && k == g->m && i < g->m) {          /* boundary column u */
        *Up = X->bu_U + di * uc;
        *Vp = X->bu_V + dk * vc;
    } else if (g->brem && i == g->m && k < g->m) {   /* boundary row v^T */
        *Up = X->bv_U + di * uc;
        *Vp = X->bv_V + dk * vc;
    } else {
        *Up = X->U + di * uc;
        *Vp = X->V + dk * vc;
    }
}

/* Dense tile (i,i): column-major d_i x d_i, ld d_i. */
static const float *dense_tile(const orc_geo *g, int64_t i) {
    const orc_mat *X = g->X;
    if (g->brem && i == g->m) return X->gamma;
    return X->D + i * X->b * X->b;
}

/* Value of stored X at (row a of tile i, column c of tile k). */
static double tile_entry(const orc_geo *g, int64_t i, int64_t k, int64_t a, int64_t c) {
    const orc_mat *X = g->X;
    int64_t di = tdim(g, i, X->rows), dk = tdim(g, k, X->cols);
    if (is_dense_tile(g, i, k)) return ORC_MUTATE == 1 ? 0.0 : (double)dense_tile(g, i)[a + c * di];
    int64_t r = rank_of(g, i, k);
    if (r == 0) return 0.0;
    const float *Up, *Vp;
    tile_factors(g, i, k, &Up, &Vp);
    double s = 0.0;
    for (int64_t t = 0; t < r; t++) {
        int64_t vi = ORC_MUTATE == 3 ? (t + c * r) % (dk * r) : c + t * dk;
        s += (double)Up[a + t * di] * (double)Vp[vi];
    }
    return s;
}

/* Row `row` of the stored matrix X, all columns, into out[0..cols). */
static void stored_row(const orc_geo *g, int64_t row, double *out) {
    const orc_mat *X = g->X;
    if (X->kind == 1) {
        for (int64_t c = 0; c < X->cols; c++) out[c] = (double)X->dense[row + c * X->ld];
        return;
    }
    int64_t i = row / X->b, a = row % X->b;
    for (int64_t k = 0; k < g->ntc; k++) {
        int64_t dk = tdim(g, k, X->cols);
        for (int64_t c = 0; c < dk; c++) out[k * X->b + c] = tile_entry(g, i, k, a, c);
    }
}

/* Column `col` of the stored matrix X, all rows, into out[0..rows). */
static void stored_col(const orc_geo *g, int64_t col, double *out) {
    const orc_mat *X = g->X;
    if (X->kind == 1) {
        for (int64_t r = 0; r < X->rows; r++) out[r] = (double)X->dense[r + col * X->ld];
        return;
    }
    int64_t k = col / X->b, c = col % X->b;
    for (int64_t i = 0; i < g->ntr; i++) {
        int64_t di = tdim(g, i, X->rows);
        for (int64_t a = 0; a < di; a++) out[i * X->b + a] = tile_entry(g, i, k, a, c);
    }
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Validate a descriptor and its ranks; 0 when valid. */
int orc_check(const orc_mat *X) {
    orc_geo g;
    int rc = geo_init(&g, X);
    geo_free(&g);
    return rc;
}

/* Dense tile (ti, tk) of op(X) into out (column-major, leading dimension ld). */
int orc_expand_tile(const orc_mat *X, int op, int64_t ti, int64_t tk, double *out, int64_t ld) {
    orc_geo g;
    int rc = geo_init(&g, X);
    if (rc) { geo_free(&g); return rc; }
    if (X->kind != 0) { geo_free(&g); return ORC_BAD_ARG; }
    int64_t si = op ? tk : ti, sk = op ? ti : tk;   /* stored tile */
    int64_t di = tdim(&g, si, X->rows), dk = tdim(&g, sk, X->cols);
    for (int64_t a = 0; a < di; a++)
        for (int64_t c = 0; c < dk; c++) {
            double v = tile_entry(&g, si, sk, a, c);
            if (op) out[c + a * ld] = v; else out[a + c * ld] = v;
        }
    geo_free(&g);
    return ORC_OK;
}

/*
 * Output block C[rows[p], cols[q]] for p < nr, q < nc:
 *   Cout[p + q*nr] = alpha * sum_t op(A)[rows[p], t] * op(B)[t, cols[q]] + beta * Cin[p + q*nr]
 * with the sum over t ascending. Cin is not read when beta == 0; the operands
 * are not read when alpha == 0.
 */
int orc_gemm_block(int opA, int opB, double alpha, const orc_mat *A, const orc_mat *B, double beta,
                   const int64_t *rows, int64_t nr, const int64_t *cols, int64_t nc,
                   const float *Cin, double *Cout) {
    if (nr < 0 || nc < 0 || (nr && !rows) || (nc && !cols) || !Cout) return ORC_BAD_ARG;
    int64_t Ar = opA ? A->cols : A->rows, Ak = opA ? A->rows : A->cols;
    int64_t Bk = opB ? B->cols : B->rows, Bc = opB ? B->rows : B->cols;
    if (Ak != Bk) return ORC_BAD_ARG;
    for (int64_t p = 0; p < nr; p++) if (rows[p] < 0 || rows[p] >= Ar) return ORC_BAD_ARG;
    for (int64_t q = 0; q < nc; q++) if (cols[q] < 0 || cols[q] >= Bc) return ORC_BAD_ARG;
    if (beta != 0.0 && !Cin && nr && nc) return ORC_BAD_ARG;
    if (ORC_MUTATE == 4) beta = -beta;
    int64_t K = Ak;
    if (alpha == 0.0) {
        for (int64_t q = 0; q < nc; q++)
            for (int64_t p = 0; p < nr; p++)
                Cout[p + q * nr] = beta != 0.0 ? beta * (double)Cin[p + q * nr] : 0.0;
        return ORC_OK;
    }
    orc_geo ga, gb;
    int rc = geo_init(&ga, A);
    if (!rc) rc = geo_init(&gb, B); else memset(&gb, 0, sizeof gb);
    if (rc) { geo_free(&ga); geo_free(&gb); return rc; }
    double *Ar_ = (double *)malloc(sizeof(double) * (size_t)(nr * K + 1));
    double *Bc_ = (double *)malloc(sizeof(double) * (size_t)(nc * K + 1));
    if (!Ar_ || !Bc_) { free(Ar_); free(Bc_); geo_free(&ga); geo_free(&gb); return ORC_NO_MEMORY; }
    /* rows of op(A): row r of A, or column r of A when op(A) = A^T */
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t p = 0; p < nr; p++) {
        if (opA) stored_col(&ga, rows[p], Ar_ + p * K);
        else stored_row(&ga, rows[p], Ar_ + p * K);
    }
    /* columns of op(B): column c of B, or row c of B when op(B) = B^T */
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t q = 0; q < nc; q++) {
        if (opB) stored_row(&gb, cols[q], Bc_ + q * K);
        else stored_col(&gb, cols[q], Bc_ + q * K);
    }
    /* entries: independent fp64 dot products, each summed in ascending t */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < nr; p++) {
        const double *a = Ar_ + p * K;
        int64_t q = 0;
        for (; q + 4 <= nc; q += 4) {
            const double *b0 = Bc_ + q * K, *b1 = b0 + K, *b2 = b1 + K, *b3 = b2 + K;
            double s0 = 0, s1 = 0, s2 = 0, s3 = 0;
            for (int64_t t = 0; t < K; t++) {
                double x = a[t];
                s0 += x * b0[t]; s1 += x * b1[t]; s2 += x * b2[t]; s3 += x * b3[t];
            }
            double s[4] = {s0, s1, s2, s3};
            for (int u = 0; u < 4; u++) {
                int64_t o = p + (q + u) * nr;
                Cout[o] = alpha * s[u] + (beta != 0.0 ? beta * (double)Cin[o] : 0.0);
            }
        }
        for (; q < nc; q++) {
            const double *b0 = Bc_ + q * K;
            double s0 = 0;
            for (int64_t t = 0; t < K; t++) s0 += a[t] * b0[t];
            int64_t o = p + q * nr;
            Cout[o] = alpha * s0 + (beta != 0.0 ? beta * (double)Cin[o] : 0.0);
        }
    }
    free(Ar_);
    free(Bc_);
    geo_free(&ga);
    geo_free(&gb);
    return ORC_OK;
}
