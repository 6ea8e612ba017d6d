/*
 * CPU oracle for CSR SpMM:  C = alpha * A * B + beta * C0.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: it is used by the tests, by the smoke check and by the
 * benchmark's CPU-baseline leg, and by nothing else.  It shares no code,
 * header or constant with the CUDA library.
 *
 * What it computes (oxicuda-sparse, ops/spmm.rs):
 *   - module doc and `spmm` doc comment: C = alpha * A * B + beta * C, A an
 *     m x k CSR matrix (row_ptr, col_idx, values), B a dense k x n matrix and
 *     C a dense m x n matrix, both row-major with leading dimensions;
 *   - device-test oracle `cpu_spmm`: per row, one accumulator per output
 *     column, summed over the row's stored entries in CSR order in f64, then
 *     alpha * acc + beta * C0;
 *   - CPU test reference `cpu_csr_spmm`: B addressed as B[col * ldb + c].
 *
 * Readings where the page is silent or departs from the arithmetic
 * (the conventions of dense BLAS):
 *   - beta == 0: C0 is not read (NaN/Inf in C0 do not propagate);
 *   - alpha == 0: A and B are not read; the result is beta * C0 (+0 if beta == 0);
 *   - k == 0 or an empty row: the accumulator stays +0, so the row is
 *     alpha * 0 + beta * C0;
 *   - duplicate column indices each contribute; explicit zeros multiply.
 *
 * Products of two binary32 numbers are exact in binary64, so for f32 inputs
 * the only rounding is in the f64 running sums.
 *
 * Every call also returns, per output, the error-bound scale
 *   bound = |alpha| * sum_p |a_p| * |b_{col_p, c}| + |beta| * |C0|
 * (the second term only when beta != 0), used by the parity tests.
 *
 * Plain loops, no blocking or reordering; single-threaded.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARGS -1
#define ORACLE_BAD_CSR -2
#define ORACLE_NO_MEMORY -3

/* Element i of an array of binary32 (esize 4) or binary64 (esize 8), widened. */
static double load(const void *p, int64_t i, int esize)
{
    if (esize == 4) return (double)((const float *)p)[i];
    return ((const double *)p)[i];
}

/* CSR structure check: row_ptr[0] == 0, non-decreasing, row_ptr[m] == nnz,
 * 0 <= col_idx[p] < k for every stored entry. */
int oracle_csr_check(int64_t m, int64_t k, int64_t nnz, const int32_t *row_ptr,
                     const int32_t *col_idx)
{
    if (m < 0 || k < 0 || nnz < 0 || !row_ptr) return ORACLE_BAD_ARGS;
    if (row_ptr[0] != 0 || (int64_t)row_ptr[m] != nnz) return ORACLE_BAD_CSR;
    for (int64_t i = 0; i < m; ++i)
        if (row_ptr[i + 1] < row_ptr[i]) return ORACLE_BAD_CSR;
    for (int64_t p = 0; p < nnz; ++p)
        if (col_idx[p] < 0 || (int64_t)col_idx[p] >= k) return ORACLE_BAD_CSR;
    return ORACLE_OK;
}

/*
 * out[r * ldo + c] = alpha * sum_{p in row i} values[p] * B[col_idx[p] * ldb + c]
 *                    + beta * C0[i * ldc + c]
 * for the rows i = rows[r], r < nrows (all rows 0..m-1 in order when rows is
 * NULL) and every column c < n.  bound (may be NULL) gets the error-bound
 * scale described above, with the same layout.
 * esize is the element size of values, B and C0: 4 (binary32) or 8 (binary64).
 */
int oracle_spmm(int esize, int64_t m, int64_t k, int64_t n, double alpha,
                const int32_t *row_ptr, const int32_t *col_idx, const void *values,
                const void *B, int64_t ldb, double beta, const void *C0, int64_t ldc,
                const int64_t *rows, int64_t nrows, double *out, double *bound, int64_t ldo)
{
    if ((esize != 4 && esize != 8) || m < 0 || k < 0 || n < 0 || ldo < n) return ORACLE_BAD_ARGS;
    if (!rows) nrows = m;
    if (nrows <= 0 || n == 0) return ORACLE_OK;
    if (beta != 0.0 && (!C0 || ldc < n)) return ORACLE_BAD_ARGS;
    if (alpha != 0.0 && (!row_ptr || ldb < n)) return ORACLE_BAD_ARGS;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= m) return ORACLE_BAD_ARGS;
        if (alpha == 0.0) continue;
        if (row_ptr[i + 1] < row_ptr[i]) return ORACLE_BAD_CSR;
        for (int64_t p = row_ptr[i]; p < (int64_t)row_ptr[i + 1]; ++p)
            if (col_idx[p] < 0 || (int64_t)col_idx[p] >= k) return ORACLE_BAD_CSR;
    }

    double *acc = (double *)malloc(sizeof(double) * (size_t)n);
    double *absacc = (double *)malloc(sizeof(double) * (size_t)n);
    if (!acc || !absacc) {
        free(acc);
        free(absacc);
        return ORACLE_NO_MEMORY;
    }

    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        double *o = out + r * ldo;
        double *bd = bound ? bound + r * ldo : NULL;

        if (alpha == 0.0) {                      /* A and B not referenced */
            for (int64_t c = 0; c < n; ++c) {
                double c0 = (beta == 0.0) ? 0.0 : load(C0, i * ldc + c, esize);
                o[c] = (beta == 0.0) ? 0.0 : beta * c0;
                if (bd) bd[c] = fabs(beta) * fabs(c0);
            }
            continue;
        }

        for (int64_t c = 0; c < n; ++c) {
            acc[c] = 0.0;
            absacc[c] = 0.0;
        }
        for (int64_t p = row_ptr[i]; p < (int64_t)row_ptr[i + 1]; ++p) {
            int64_t j = col_idx[p];
            double a = load(values, p, esize);
            for (int64_t c = 0; c < n; ++c) {
                double b = load(B, j * ldb + c, esize);
                acc[c] += a * b;
                absacc[c] += fabs(a) * fabs(b);
            }
        }
        for (int64_t c = 0; c < n; ++c) {
            double v = alpha * acc[c];
            double e = fabs(alpha) * absacc[c];
            if (beta != 0.0) {                   /* C0 read only when beta != 0 */
                double c0 = load(C0, i * ldc + c, esize);
                v += beta * c0;
                e += fabs(beta) * fabs(c0);
            }
            o[c] = v;
            if (bd) bd[c] = e;
        }
    }
    free(acc);
    free(absacc);
    return ORACLE_OK;
}

/*
 * The squared chain, for a square m x m CSR matrix A (the SEACells kernel
 * matrix K of the bixverse page, whose Frank-Wolfe kernels consume
 * K^2 B, the output of `k_squared_matmul`, module doc):
 *
 *   out[r * ldo + c] = alpha * (A (A B))[i, c] + beta * C0[i * ldc + c],
 *   i = rows[r] (all rows in order when rows is NULL), c < n.
 *
 * Plain definition, written out: for each entry (i, j) of row i, row j of the
 * intermediate T = A B is formed in binary64 from row j's entries (T is never
 * rounded to the input precision), and the output row accumulates
 * a_ij * T[j, c] in CSR order.  alpha == 0: A and B are not read; beta == 0:
 * C0 is not read (as for the single product).
 *
 * bound = |alpha| * sum_j |a_ij| * sum_l |a_jl| * |B[l, c]| + |beta| * |C0|,
 * the same scale as the single product, with |A| |A| |B| in place of |A| |B|.
 */
int oracle_spmm_squared(int esize, int64_t m, int64_t n, double alpha,
                        const int32_t *row_ptr, const int32_t *col_idx, const void *values,
                        const void *B, int64_t ldb, double beta, const void *C0, int64_t ldc,
                        const int64_t *rows, int64_t nrows, double *out, double *bound,
                        int64_t ldo)
{
    if ((esize != 4 && esize != 8) || m < 0 || n < 0 || ldo < n) return ORACLE_BAD_ARGS;
    if (!rows) nrows = m;
    if (nrows <= 0 || n == 0) return ORACLE_OK;
    if (beta != 0.0 && (!C0 || ldc < n)) return ORACLE_BAD_ARGS;
    if (alpha != 0.0) {
        if (!row_ptr || ldb < n) return ORACLE_BAD_ARGS;
        if (oracle_csr_check(m, m, (int64_t)row_ptr[m], row_ptr, col_idx) != ORACLE_OK)
            return ORACLE_BAD_CSR;
    }
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= m) return ORACLE_BAD_ARGS;
    }

    double *acc = (double *)malloc(sizeof(double) * (size_t)n);
    double *absacc = (double *)malloc(sizeof(double) * (size_t)n);
    double *t = (double *)malloc(sizeof(double) * (size_t)n);      /* row j of A B */
    double *abst = (double *)malloc(sizeof(double) * (size_t)n);   /* row j of |A| |B| */
    if (!acc || !absacc || !t || !abst) {
        free(acc);
        free(absacc);
        free(t);
        free(abst);
        return ORACLE_NO_MEMORY;
    }

    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        double *o = out + r * ldo;
        double *bd = bound ? bound + r * ldo : NULL;

        if (alpha == 0.0) {                      /* A and B not referenced */
            for (int64_t c = 0; c < n; ++c) {
                double c0 = (beta == 0.0) ? 0.0 : load(C0, i * ldc + c, esize);
                o[c] = (beta == 0.0) ? 0.0 : beta * c0;
                if (bd) bd[c] = fabs(beta) * fabs(c0);
            }
            continue;
        }

        for (int64_t c = 0; c < n; ++c) {
            acc[c] = 0.0;
            absacc[c] = 0.0;
        }
        for (int64_t p = row_ptr[i]; p < (int64_t)row_ptr[i + 1]; ++p) {
            int64_t j = col_idx[p];
            double a = load(values, p, esize);
            for (int64_t c = 0; c < n; ++c) {
                t[c] = 0.0;
                abst[c] = 0.0;
            }
            for (int64_t q = row_ptr[j]; q < (int64_t)row_ptr[j + 1]; ++q) {
                int64_t l = col_idx[q];
                double aj = load(values, q, esize);
                for (int64_t c = 0; c < n; ++c) {
                    double b = load(B, l * ldb + c, esize);
                    t[c] += aj * b;
                    abst[c] += fabs(aj) * fabs(b);
                }
            }
            for (int64_t c = 0; c < n; ++c) {
                acc[c] += a * t[c];
                absacc[c] += fabs(a) * abst[c];
            }
        }
        for (int64_t c = 0; c < n; ++c) {
            double v = alpha * acc[c];
            double e = fabs(alpha) * absacc[c];
            if (beta != 0.0) {                   /* C0 read only when beta != 0 */
                double c0 = load(C0, i * ldc + c, esize);
                v += beta * c0;
                e += fabs(beta) * fabs(c0);
            }
            o[c] = v;
            if (bd) bd[c] = e;
        }
    }
    free(acc);
    free(absacc);
    free(t);
    free(abst);
    return ORACLE_OK;
}

/*
 * The Frank-Wolfe gradient scan of the B update (bixverse page,
 * seacells_kernels.rs: `fw_argmin_b` doc comment and the CPU reference of its
 * tests, `cpu_fw_argmin_b`).  With K2B and T2 = K^2 A^T given as n x k CSR,
 * t1 = A A^T as k x k CSR and B as n x k CSR:
 *
 *   G[i, c] = sum_m K2B[i, m] * t1[m, c] - T2[i, c]
 *   min_val[c] = min_i G[i, c],  min_idx[c] = the lowest i attaining it
 *   gap = sum over stored entries (i, c) of B of B[i, c] * G[i, c]
 *
 * Rows are scanned in increasing i with a strict <, starting from the
 * largest finite value and index 0, as the page's CPU scan does (so n == 0,
 * or a column whose G never falls below that start, reports it with index
 * 0).  Stored entries each contribute (duplicates add).  Everything is
 * accumulated in binary64.
 *
 * Bound scales (for the parity tests): gbound[i, c] = sum_m |K2B[i, m]| *
 * |t1[m, c]| + |T2[i, c]| bounds the rounding of G[i, c]; col_scale[c] is its
 * maximum over i; gap_bound = sum over B's entries of |B[i, c]| * gbound[i, c].
 */
static void fw_gradient_row(int esize, int64_t k, int64_t i,
                            const int32_t *k2b_rp, const int32_t *k2b_ci, const void *k2b_v,
                            const int32_t *t1_rp, const int32_t *t1_ci, const void *t1_v,
                            const int32_t *t2_rp, const int32_t *t2_ci, const void *t2_v,
                            double *g, double *gb)
{
    for (int64_t c = 0; c < k; ++c) {
        g[c] = 0.0;
        gb[c] = 0.0;
    }
    for (int64_t p = k2b_rp[i]; p < (int64_t)k2b_rp[i + 1]; ++p) {
        int64_t m = k2b_ci[p];
        double v = load(k2b_v, p, esize);
        for (int64_t q = t1_rp[m]; q < (int64_t)t1_rp[m + 1]; ++q) {
            int64_t c = t1_ci[q];
            double t = load(t1_v, q, esize);
            g[c] += v * t;
            gb[c] += fabs(v) * fabs(t);
        }
    }
    for (int64_t q = t2_rp[i]; q < (int64_t)t2_rp[i + 1]; ++q) {
        int64_t c = t2_ci[q];
        double t = load(t2_v, q, esize);
        g[c] -= t;
        gb[c] += fabs(t);
    }
}

static int fw_check(int64_t n, int64_t k, const int32_t *k2b_rp, const int32_t *k2b_ci,
                    const int32_t *t1_rp, const int32_t *t1_ci, const int32_t *t2_rp,
                    const int32_t *t2_ci)
{
    if (!k2b_rp || !t1_rp || !t2_rp) return ORACLE_BAD_ARGS;
    if (oracle_csr_check(n, k, (int64_t)k2b_rp[n], k2b_rp, k2b_ci) != ORACLE_OK ||
        oracle_csr_check(k, k, (int64_t)t1_rp[k], t1_rp, t1_ci) != ORACLE_OK ||
        oracle_csr_check(n, k, (int64_t)t2_rp[n], t2_rp, t2_ci) != ORACLE_OK)
        return ORACLE_BAD_CSR;
    return ORACLE_OK;
}

/* G rows: g[r * k + c] = G[rows[r], c] and gbound likewise (rows NULL: all). */
int oracle_fw_gradient(int esize, int64_t n, int64_t k,
                       const int32_t *k2b_rp, const int32_t *k2b_ci, const void *k2b_v,
                       const int32_t *t1_rp, const int32_t *t1_ci, const void *t1_v,
                       const int32_t *t2_rp, const int32_t *t2_ci, const void *t2_v,
                       const int64_t *rows, int64_t nrows, double *g, double *gbound)
{
    if ((esize != 4 && esize != 8) || n < 0 || k < 0) return ORACLE_BAD_ARGS;
    int rc = fw_check(n, k, k2b_rp, k2b_ci, t1_rp, t1_ci, t2_rp, t2_ci);
    if (rc != ORACLE_OK) return rc;
    if (!rows) nrows = n;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= n) return ORACLE_BAD_ARGS;
        fw_gradient_row(esize, k, i, k2b_rp, k2b_ci, k2b_v, t1_rp, t1_ci, t1_v, t2_rp, t2_ci,
                        t2_v, g + r * k, gbound + r * k);
    }
    return ORACLE_OK;
}

int oracle_fw_argmin(int esize, int64_t n, int64_t k,
                     const int32_t *k2b_rp, const int32_t *k2b_ci, const void *k2b_v,
                     const int32_t *t1_rp, const int32_t *t1_ci, const void *t1_v,
                     const int32_t *t2_rp, const int32_t *t2_ci, const void *t2_v,
                     const int32_t *b_rp, const int32_t *b_ci, const void *b_v,
                     double *min_val, int64_t *min_idx, double *col_scale, double *gap,
                     double *gap_bound)
{
    if ((esize != 4 && esize != 8) || n < 0 || k < 0 || !gap || !gap_bound) return ORACLE_BAD_ARGS;
    if (k > 0 && (!min_val || !min_idx || !col_scale)) return ORACLE_BAD_ARGS;
    int rc = fw_check(n, k, k2b_rp, k2b_ci, t1_rp, t1_ci, t2_rp, t2_ci);
    if (rc != ORACLE_OK) return rc;
    if (!b_rp || oracle_csr_check(n, k, (int64_t)b_rp[n], b_rp, b_ci) != ORACLE_OK)
        return ORACLE_BAD_CSR;
    /* the start of the scan: the largest finite value of the element type */
    const double start = (esize == 4) ? 3.4028234663852886e38 : 1.7976931348623157e308;
    for (int64_t c = 0; c < k; ++c) {
        min_val[c] = start;
        min_idx[c] = 0;
        col_scale[c] = 0.0;
    }
    *gap = 0.0;
    *gap_bound = 0.0;
    double *g = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    double *gb = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    if (!g || !gb) {
        free(g);
        free(gb);
        return ORACLE_NO_MEMORY;
    }
    for (int64_t i = 0; i < n; ++i) {
        fw_gradient_row(esize, k, i, k2b_rp, k2b_ci, k2b_v, t1_rp, t1_ci, t1_v, t2_rp, t2_ci,
                        t2_v, g, gb);
        for (int64_t r = b_rp[i]; r < (int64_t)b_rp[i + 1]; ++r) {
            int64_t c = b_ci[r];
            double b = load(b_v, r, esize);
            *gap += b * g[c];
            *gap_bound += fabs(b) * gb[c];
        }
        for (int64_t c = 0; c < k; ++c) {
            if (g[c] < min_val[c]) {             /* strict: the lowest row wins a tie */
                min_val[c] = g[c];
                min_idx[c] = i;
            }
            if (gb[c] > col_scale[c]) col_scale[c] = gb[c];
        }
    }
    free(g);
    free(gb);
    return ORACLE_OK;
}

/*
 * ILU(0): the incomplete LU factorisation with zero fill-in of the oxicuda
 * preconditioner page (preconditioner/ilu0.rs: module doc, `ilu0`, the host
 * row factorisation and the level analysis).  A is square, CSR with column
 * indices strictly ascending within each row.
 *
 * Levels: depth(i) = 1 + max depth(k) over the stored k < i of row i (0 when
 * there is none); rows are factored level by level, and within a level in
 * increasing index order.
 *
 * The elimination is Gaussian elimination in its row-oriented (IKJ) form,
 * confined to A's pattern.  Row i is brought to its final value by
 * subtracting multiples of the already factored rows k < i that it stores,
 * k ascending: l_ik = a_ik / u_kk, then a_ij -= l_ik * u_kj for every j > k
 * stored in both rows (a j outside row i's pattern would be fill-in, which
 * ILU(0) drops).  A zero or absent u_kk is a singular pivot.  Each operation
 * is one rounded divide, multiply or subtract in the element type (binary32
 * or binary64), as on the page (no fused multiply-add; this file is compiled
 * without contraction); every a_ij receives its updates in ascending k, so a
 * correct implementation reproduces it bit for bit.  L is the strictly
 * lower part with a unit diagonal, U the rest.
 *
 * Bookkeeping: diag[r] is where row r stores its diagonal (-1 if nowhere);
 * slot[c] is where the row being eliminated stores column c (-1 if it does
 * not), filled before the row and cleared after it.
 */
#define ORACLE_SINGULAR -4

#define ILU0_ELIMINATE(NAME, T)                                                          \
    static int NAME(int64_t n, const int32_t *rp, const int32_t *ci, T *v,               \
                    const int64_t *order, const int64_t *diag, int64_t *slot)            \
    {                                                                                    \
        for (int64_t r = 0; r < n; ++r) {                                                \
            const int64_t i = order[r];                                                  \
            const int64_t lo = rp[i], hi = rp[i + 1];                                    \
            int rc = ORACLE_OK;                                                          \
            for (int64_t p = lo; p < hi; ++p) slot[ci[p]] = p;                           \
            for (int64_t p = lo; p < hi && ci[p] < i; ++p) {                             \
                const int64_t k = ci[p];                                                 \
                const int64_t pk = diag[k];                                              \
                if (pk < 0 || v[pk] == (T)0) {                                           \
                    rc = ORACLE_SINGULAR;                                                \
                    break;                                                               \
                }                                                                        \
                const T l_ik = v[p] / v[pk];                                             \
                v[p] = l_ik;                                                             \
                for (int64_t q = pk + 1; q < (int64_t)rp[k + 1]; ++q) {                  \
                    const int64_t t = slot[ci[q]];                                       \
                    if (t < 0) continue;                /* fill-in: dropped */           \
                    const T prod = l_ik * v[q];                                          \
                    v[t] = v[t] - prod;                                                  \
                }                                                                        \
            }                                                                            \
            for (int64_t p = lo; p < hi; ++p) slot[ci[p]] = -1;                          \
            if (rc != ORACLE_OK) return rc;                                              \
        }                                                                                \
        return ORACLE_OK;                                                                \
    }
ILU0_ELIMINATE(ilu0_eliminate_f32, float)
ILU0_ELIMINATE(ilu0_eliminate_f64, double)

/* depth[i] for every row (the page's level analysis); returns the level count. */
int64_t oracle_ilu0_levels(int64_t n, const int32_t *rp, const int32_t *ci, int64_t *depth)
{
    int64_t max_depth = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t d = 0;
        for (int64_t p = rp[i]; p < (int64_t)rp[i + 1]; ++p) {
            const int64_t j = ci[p];
            if (j < i && depth[j] + 1 > d) d = depth[j] + 1;
        }
        depth[i] = d;
        if (d > max_depth) max_depth = d;
    }
    return n > 0 ? max_depth + 1 : 0;
}

/* Factor in place; depth (may be NULL) gets each row's level.  Returns
 * ORACLE_OK, ORACLE_SINGULAR, or ORACLE_BAD_ARGS / ORACLE_BAD_CSR. */
int oracle_ilu0(int esize, int64_t n, const int32_t *rp, const int32_t *ci, void *values,
                int64_t *depth)
{
    if ((esize != 4 && esize != 8) || n <= 0 || !rp || !values) return ORACLE_BAD_ARGS;
    if (oracle_csr_check(n, n, (int64_t)rp[n], rp, ci) != ORACLE_OK) return ORACLE_BAD_CSR;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t p = rp[i] + 1; p < (int64_t)rp[i + 1]; ++p)
            if (ci[p] <= ci[p - 1]) return ORACLE_BAD_CSR;   /* strictly ascending */
    int64_t *d = depth ? depth : (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
    int64_t *order = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
    int64_t *diag = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
    int64_t *slot = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
    int64_t *start = NULL;
    int rc = ORACLE_NO_MEMORY;
    if (!d || !order || !diag || !slot) goto done;
    const int64_t nlev = oracle_ilu0_levels(n, rp, ci, d);
    /* rows grouped by level, increasing index within a level (counting sort) */
    start = (int64_t *)calloc((size_t)nlev + 1, sizeof(int64_t));
    if (!start) goto done;
    for (int64_t i = 0; i < n; ++i) start[d[i] + 1]++;
    for (int64_t l = 0; l < nlev; ++l) start[l + 1] += start[l];
    for (int64_t i = 0; i < n; ++i) order[start[d[i]]++] = i;
    for (int64_t i = 0; i < n; ++i) {
        diag[i] = -1;
        slot[i] = -1;
        for (int64_t p = rp[i]; p < (int64_t)rp[i + 1]; ++p)
            if (ci[p] == i) diag[i] = p;
    }
    rc = (esize == 4) ? ilu0_eliminate_f32(n, rp, ci, (float *)values, order, diag, slot)
                      : ilu0_eliminate_f64(n, rp, ci, (double *)values, order, diag, slot);
done:
    if (!depth) free(d);
    free(order);
    free(diag);
    free(slot);
    free(start);
    return rc;
}
