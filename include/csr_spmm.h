/*
 * csr_spmm.h -- C ABI of the GB300 (sm_103a) CSR SpMM library.
 *
 * Operation (oxicuda-sparse, ops/spmm.rs: module doc and `spmm` doc comment):
 *
 *     C = alpha * A * B + beta * C
 *
 * A is an m x k sparse matrix in CSR form: row_ptr (int32, m + 1 entries),
 * col_idx (int32, nnz entries) and values (nnz entries), nnz = row_ptr[m].
 * B is a dense k x n matrix and C a dense m x n matrix, both row-major with
 * leading dimensions ldb and ldc (element (r, c) of B lives at B[r * ldb + c]).
 * The page's `spmm` takes (handle, alpha, A, B, beta, C) and launches with the
 * arguments (row_ptr, col_idx, values, B, C, alpha, beta, m, n, ldb, ldc) on
 * the handle's stream; this ABI passes the same quantities flat, plus k and the
 * stream.
 *
 * Conventions (the page always reads C and returns early when k == 0; these
 * are the readings this library implements, those of dense BLAS):
 *   - beta == 0: C is write-only; its previous contents (even NaN/Inf) are
 *     never read.
 *   - alpha == 0: A and B are not read; C = beta * C (C = 0 when beta == 0).
 *   - k == 0 (every row empty): C = beta * C.  An empty row i gives
 *     C[i, :] = beta * C[i, :].
 *   - m == 0 or n == 0: nothing is done.
 *   - Duplicate column indices within a row each contribute; explicit zeros
 *     are multiplied like any other entry.
 *   - Results are deterministic: the same inputs give bit-identical C on every
 *     call (no floating-point atomics; every sum has a fixed order).
 *
 * Memory and ownership: every array argument is a DEVICE pointer on the
 * handle's device, owned by the caller and not retained after the call
 * returns.  The handle owns its scratch memory (row bins, long-row partial
 * sums) and grows it on demand; growth calls cudaMalloc/cudaFree, which
 * synchronise the device, so reserve it first (spmm_reserve) when the call
 * will be captured in a CUDA graph.  C must not overlap A or B.
 *
 * Asynchrony: the products are enqueued on `stream` (a cudaStream_t passed as
 * void*; NULL means the legacy default stream) and return without
 * synchronising.  Launch errors are returned; a fault inside a kernel
 * surfaces at the caller's next synchronisation.  A handle may be used by one
 * stream at a time (its scratch is shared by its calls).
 *
 * CSR contents are a precondition: row_ptr[0] == 0, row_ptr non-decreasing,
 * 0 <= col_idx[p] < k.  They are not checked on the product path (nor are
 * they on the page); spmm_csr_check verifies them on the device.
 */
#ifndef CSR_SPMM_H
#define CSR_SPMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  The page's error kinds map as: DimensionMismatch ->
 * SPMM_ERR_DIMENSION_MISMATCH, InvalidArgument -> SPMM_ERR_INVALID_ARGUMENT,
 * Cuda -> SPMM_ERR_CUDA (oxicuda-sparse, ops/spmm.rs, `spmm` "Errors"). */
typedef enum {
    SPMM_OK = 0,
    SPMM_ERR_INVALID_ARGUMENT = 1,   /* bad handle, negative or oversize m/k/n, wrong device */
    SPMM_ERR_DIMENSION_MISMATCH = 2, /* ldb < max(1, n) or ldc < max(1, n) */
    SPMM_ERR_NULL_POINTER = 3,       /* a pointer that the call must dereference is NULL */
    SPMM_ERR_UNSUPPORTED_DEVICE = 4, /* device is not compute capability 10.x / sm_103 family */
    SPMM_ERR_ALLOC = 5,              /* scratch allocation failed */
    SPMM_ERR_CUDA = 6,               /* a CUDA runtime call or kernel launch failed */
    SPMM_ERR_INVALID_CSR = 7,        /* spmm_csr_check found a malformed CSR structure */
    SPMM_ERR_TOO_LARGE = 8           /* beyond the fixed limits of spmm_csr_f32_noalloc */
} spmm_status_t;

typedef struct spmm_handle_s *spmm_handle_t;

/* Create a handle for `device` (a CUDA ordinal).  Queries the SM count and
 * L2 size used to size grids and column panels.  Does not change the current
 * device.  *h is set to NULL on failure. */
spmm_status_t spmm_create(spmm_handle_t *h, int device);

/* Release the handle and its scratch.  Synchronises the handle's device.
 * NULL is accepted and ignored. */
spmm_status_t spmm_destroy(spmm_handle_t h);

/* Grow the handle's scratch for products with up to m rows and n columns of
 * the given element size (4 or 8 bytes), so that later calls of that size
 * allocate nothing.  Synchronous. */
spmm_status_t spmm_reserve(spmm_handle_t h, int64_t m, int64_t n, int elem_size);

/* C = alpha * A * B + beta * C in binary32 (oxicuda-sparse, ops/spmm.rs, `spmm`
 * with T = f32).  Up to m = 2048 rows the product is one kernel launch and
 * uses no handle scratch; larger products bin the rows in a pre-pass first.
 * Arguments as described at the top of this file:
 *   row_ptr [m+1], col_idx [nnz], values [nnz]   CSR of A (m x k)
 *   B  [k rows, stride ldb]   dense, row-major, only columns 0..n-1 are read
 *   C  [m rows, stride ldc]   dense, row-major, columns 0..n-1 are written
 * Requires m, k, n >= 0, m < 2^31 - 1, k <= 2^31 - 1, max(1, n) <= ldb <=
 * 2^31 - 1 (SPMM_ERR_INVALID_ARGUMENT above), ldc >= max(1, n); the current
 * device must be the handle's device.
 * Pointers may be NULL only where the conventions above say the array is not
 * read (A and B when alpha == 0 or k == 0; everything when m == 0 or n == 0).
 * The library cannot see nnz, so col_idx and values must be valid addresses
 * whenever A is read, even for nnz == 0. */
spmm_status_t spmm_csr_f32(spmm_handle_t h, float alpha,
                           const int32_t *row_ptr, const int32_t *col_idx, const float *values,
                           int64_t m, int64_t k,
                           const float *B, int64_t ldb, int64_t n,
                           float beta, float *C, int64_t ldc, void *stream);

/* Same in binary64 (the page's `spmm` with T = f64). */
spmm_status_t spmm_csr_f64(spmm_handle_t h, double alpha,
                           const int32_t *row_ptr, const int32_t *col_idx, const double *values,
                           int64_t m, int64_t k,
                           const double *B, int64_t ldb, int64_t n,
                           double beta, double *C, int64_t ldc, void *stream);

/* Check the CSR structure on the device: row_ptr[0] == 0, row_ptr
 * non-decreasing, row_ptr[m] == nnz, and 0 <= col_idx[p] < k for p < nnz.
 * Reads exactly row_ptr[0..m] and col_idx[0..nnz-1].  Synchronises `stream`
 * and stores a bit mask in *host_status (0 = valid; bit 0: row_ptr[0] != 0,
 * bit 1: row_ptr decreases, bit 2: row_ptr[m] != nnz, bit 3: a column index
 * out of range).  Returns SPMM_ERR_INVALID_CSR when the mask is non-zero.
 * A debugging aid: the product entry points never run it. */
spmm_status_t spmm_csr_check(spmm_handle_t h, const int32_t *row_ptr, const int32_t *col_idx,
                             int64_t m, int64_t k, int64_t nnz, void *stream,
                             int32_t *host_status);

/* ---- The squared chain ----------------------------------------------------
 * C = alpha * A (A B) + beta * C for a square m x m CSR matrix A: the K^2 B
 * product that the SEACells Frank-Wolfe kernels of the bixverse page consume
 * (seacells_kernels.rs, module doc: the n x k output of `k_squared_matmul`,
 * with K the cells x cells kernel matrix).  Computed as two products that
 * share one row-binning pre-pass: T = A B into handle scratch (m x n, leading
 * dimension n rounded up to 16 bytes, grown with cudaMalloc like the rest of
 * the scratch), then C = alpha * A T + beta * C.  T is rounded to the element
 * type, so the result carries the rounding of both products; the parity
 * tolerance is twice that of one product, against the bound scale
 * |alpha| |A| |A| |B| + |beta| |C0|.  T is stored with the default L2 policy
 * (the single product streams C), so that the second product finds it in L2
 * when it fits.  B and C must not overlap.  Arguments, conventions (alpha ==
 * 0: C = beta * C and A, B are not read; beta == 0: C is not read; m == 0 or
 * n == 0: no-op) and errors as for spmm_csr_f32, with k = m.  A profiled call
 * reports the pre-pass in prepass_ms, the first product in rows_ms and the
 * second in long_ms.  Asynchronous on `stream`. */
spmm_status_t spmm_csr_squared_f32(spmm_handle_t h, float alpha,
                                   const int32_t *row_ptr, const int32_t *col_idx,
                                   const float *values, int64_t m,
                                   const float *B, int64_t ldb, int64_t n,
                                   float beta, float *C, int64_t ldc, void *stream);

/* Same in binary64. */
spmm_status_t spmm_csr_squared_f64(spmm_handle_t h, double alpha,
                                   const int32_t *row_ptr, const int32_t *col_idx,
                                   const double *values, int64_t m,
                                   const double *B, int64_t ldb, int64_t n,
                                   double beta, double *C, int64_t ldc, void *stream);

/* ---- Frank-Wolfe gradient scan ---------------------------------------------
 * The step after the product in the SEACells B update (bixverse page,
 * seacells_kernels.rs: `fw_argmin_b` and `reduce_argmin_blocks`).  With K2B
 * (= K^2 B) and T2 (= K^2 A^T) n x k CSR, t1 (= A A^T) k x k CSR and B n x k
 * CSR, all device arrays:
 *   G[i, c]    = sum_m K2B[i, m] * t1[m, c] - T2[i, c]   (never stored)
 *   min_val[c] = min over i of G[i, c]; min_idx[c] = the lowest i attaining it
 *   gap[0]     = sum over B's stored entries (i, c) of B[i, c] * G[i, c]
 * The scan starts from the largest finite value of the element type with
 * row 0, as the page's CPU scan does, and moves only on a strictly smaller
 * G, so n == 0 (or a column whose G never falls below the start) reports
 * that value with row 0.  Every row takes part, including rows with no K2B
 * entries (G = -T2 there).  Stored duplicates each contribute.  Results
 * are deterministic: no float atomics, and the gap is summed in binary64 in a
 * fixed order, then rounded to the element type.
 * Requires n, k >= 0 and valid CSR structures with column indices in [0, k)
 * (spmm_csr_check can verify them; the hot path does not), and columns
 * ascending within each row of every matrix, the page's convention
 * (duplicates, if any, then sit together and are added).
 * binary32 with k <= 104 runs the contraction K2B t1 on the tensor cores:
 * every value is split into two tf32 parts and each product is formed from
 * three tf32 products (hi hi, hi lo, lo hi), exact in binary32 and short of
 * the exact product by less than 2^-21 of |K2B[i, m]| |t1[m, c]|, with the
 * sums accumulated in binary32; other scans sum K2B entry by entry with
 * binary32 or binary64 fused multiply-adds.
 * Arrays may be NULL only when n == 0 (the n x k matrices) or k == 0 (t1,
 * min_val, min_idx); gap must always be valid.  Uses handle scratch, grown
 * with cudaMalloc: a dense, zero-padded copy of t1 (k rows of k rounded up to
 * 128 binary32 or 64 binary64 columns) and per-block partial minima.  Asynchronous on `stream`;
 * SPMM_ERR_CUDA on a launch failure. */
spmm_status_t spmm_fw_argmin_f32(spmm_handle_t h, int64_t n, int64_t k,
                                 const int32_t *k2b_row_ptr, const int32_t *k2b_col_idx,
                                 const float *k2b_values,
                                 const int32_t *t1_row_ptr, const int32_t *t1_col_idx,
                                 const float *t1_values,
                                 const int32_t *t2_row_ptr, const int32_t *t2_col_idx,
                                 const float *t2_values,
                                 const int32_t *b_row_ptr, const int32_t *b_col_idx,
                                 const float *b_values,
                                 float *min_val, int32_t *min_idx, float *gap, void *stream);

/* Same in binary64. */
spmm_status_t spmm_fw_argmin_f64(spmm_handle_t h, int64_t n, int64_t k,
                                 const int32_t *k2b_row_ptr, const int32_t *k2b_col_idx,
                                 const double *k2b_values,
                                 const int32_t *t1_row_ptr, const int32_t *t1_col_idx,
                                 const double *t1_values,
                                 const int32_t *t2_row_ptr, const int32_t *t2_col_idx,
                                 const double *t2_values,
                                 const int32_t *b_row_ptr, const int32_t *b_col_idx,
                                 const double *b_values,
                                 double *min_val, int32_t *min_idx, double *gap, void *stream);

/* ---- ILU(0) ------------------------------------------------------------------
 * Incomplete LU factorisation with zero fill-in of the oxicuda preconditioner
 * page (preconditioner/ilu0.rs, module doc and `factor_row_host`): A ~ L U
 * with L unit lower and U upper triangular, both in A's sparsity pattern.
 * Factored in place on `values` (device, A's n x n CSR values): afterwards the
 * strictly lower entries hold L (its unit diagonal is implicit) and the
 * diagonal and upper entries hold U; the page's (L, U) split is that reading.
 * Arithmetic as on the page: for each stored k < i of row i in CSR order,
 * a_ik = a_ik / a_kk, then a_ij = a_ij - a_ik * a_kj for each stored j > k
 * of row k that row i also stores, each a single rounded operation in the
 * element type (no fused multiply-add), so the result matches the page's host
 * reference bit for bit.  depth (optional, device [n]) receives each row's
 * dependency level (the page's level analysis: 1 + the deepest k < i stored
 * in row i, 0 if none).
 * Scheduled on the device without host synchronisation: dependency counts and
 * the lists of dependent rows are built by three small kernels, then one
 * persistent launch factors each row as soon as the rows it depends on are
 * final (the page launches one kernel per level and synchronises between
 * them).  Finished rows pass their values on through published copies in
 * handle scratch, preset to a signalling-NaN sentinel; an input value with
 * exactly the sentinel's bits is still handled, on a slower path.
 * nnz = row_ptr[n] (the library cannot read it without a
 * synchronisation).  status (device, one int32, required) is
 * zeroed, then receives SPMM_ILU0_SINGULAR if a pivot row lacks its diagonal
 * or has a zero one, and SPMM_ILU0_WAIT_TIMEOUT if a wait for a pivot row ran
 * out (every wait is bounded; neither happens on valid input).  After a
 * failure the values are partly factored.
 * Requires n >= 1 (n == 0: SPMM_ERR_INVALID_ARGUMENT, as the page), a valid
 * CSR structure with column indices strictly ascending within each row (no
 * duplicates), and no concurrent call on the same handle (it uses handle
 * scratch: 69n + n / 1024 + 4 nnz + 12 int32 words for binary32, one more
 * word per entry for binary64).  Asynchronous on `stream`. */
#define SPMM_ILU0_SINGULAR 1
#define SPMM_ILU0_WAIT_TIMEOUT 2
spmm_status_t spmm_ilu0_f32(spmm_handle_t h, int64_t n, int64_t nnz, const int32_t *row_ptr,
                            const int32_t *col_idx, float *values, int32_t *depth,
                            int32_t *status, void *stream);
spmm_status_t spmm_ilu0_f64(spmm_handle_t h, int64_t n, int64_t nnz, const int32_t *row_ptr,
                            const int32_t *col_idx, double *values, int32_t *depth,
                            int32_t *status, void *stream);

/* Persisting L2 for B.  With `bytes` > 0 (or < 0 for the device maximum,
 * about 81 MiB on GB300) the handle sets the process's
 * persisting-L2 set-aside to that size (cudaLimitPersistingL2CacheSize), and
 * every later product on the handle whose B span fits in the set-aside
 * launches with an access-policy window over B (hit ratio 1, persisting), so
 * that the streamed A entries and C stores cannot evict B rows between their
 * gathers.  Products with a larger B get no window.  bytes == 0 demotes all
 * persisting lines (cudaCtxResetPersistingL2Cache) and puts the previous
 * set-aside back; spmm_destroy does the same.  The set-aside belongs to the
 * whole CUDA context, so other kernels of the process see less L2 while it is
 * on: off by default.  Not synchronising.  SPMM_ERR_UNSUPPORTED_DEVICE if the
 * device has no persisting L2.  The pages place an access-policy window on B
 * without further detail; this is that window, made optional because GB300
 * measurements show a small gain only when B fits the set-aside. */
spmm_status_t spmm_set_l2_persistence(spmm_handle_t h, int64_t bytes);

/* ---- Analysis reuse: plans ------------------------------------------------
 * A plan holds the row bins of one sparsity structure (row_ptr of an m x k
 * matrix) for products with n columns, so that repeated products with the same
 * structure -- new values, new B, new C, as in an iterative solver that applies
 * one kernel matrix every iteration -- skip the row-binning pre-pass.  The
 * product is the same operation with the same conventions and bitwise the same
 * results as spmm_csr_f32/f64 on the same handle.  The plan owns device
 * scratch, allocated when it is created. */
typedef struct spmm_plan_s *spmm_plan_t;

/* Analyse row_ptr (device, m + 1 entries) on `stream` and create a plan for
 * m x k matrices with that structure and n-column products of elem_size (4 or
 * 8) byte elements.  Synchronises `stream` (it reads the bin counts back once).
 * The handle must outlive the plan and serve one stream at a time, as for
 * direct products.  CSR validity is the caller's precondition, as everywhere. */
spmm_status_t spmm_plan_create(spmm_handle_t h, spmm_plan_t *plan, const int32_t *row_ptr,
                               int64_t m, int64_t k, int64_t n, int elem_size, void *stream);

/* Release a plan (synchronises its device).  NULL is accepted and ignored.
 * Does not touch the handle, so it may run after spmm_destroy of the handle;
 * products on a plan need the handle alive. */
spmm_status_t spmm_plan_destroy(spmm_plan_t plan);

/* The squared chain C = alpha * A (A B) + beta * C (as spmm_csr_squared_f32,
 * the K^2 B operand of the SEACells Frank-Wolfe kernels of the bixverse page)
 * with A's structure taken from a plan made for a square A (k == m): both
 * products use the plan's bins and row order, so neither runs a pre-pass.
 * The intermediate A B lives in the scratch of the plan's handle (m x n,
 * leading dimension rounded up to 16 bytes, grown with cudaMalloc like any
 * handle scratch).  Same arguments and conventions as spmm_csr_squared_f32,
 * with m and n from the plan; the results equal spmm_csr_squared_f32's bit
 * for bit.  SPMM_ERR_INVALID_ARGUMENT if the plan is not square or was made
 * for the other element size.  Asynchronous on `stream`. */
spmm_status_t spmm_plan_csr_squared_f32(spmm_plan_t plan, float alpha,
                                        const int32_t *row_ptr, const int32_t *col_idx,
                                        const float *values, const float *B, int64_t ldb,
                                        float beta, float *C, int64_t ldc, void *stream);

/* Same in binary64. */
spmm_status_t spmm_plan_csr_squared_f64(spmm_plan_t plan, double alpha,
                                        const int32_t *row_ptr, const int32_t *col_idx,
                                        const double *values, const double *B, int64_t ldb,
                                        double beta, double *C, int64_t ldc, void *stream);

/* Change the order in which the plan's products process the rows of A (not
 * where results go): the short- and medium-row lists are re-sorted into the
 * breadth-first order of A's pattern (spmm_row_order_bfs), so that rows which
 * gather the same B rows run next to each other and share the SM's L1.  Worth
 * it for matrices whose pattern has locality that the row numbering hides, as
 * in the kNN kernel matrix that the SEACells Frank-Wolfe kernels of the
 * bixverse page apply every iteration; of no use for uniformly random
 * columns.  Long rows keep their order.  Results stay bitwise the same as
 * without the call: each row's sum does not depend on when it is computed.
 * row_ptr and col_idx are device arrays holding the structure the plan
 * analysed (row_ptr with the same values).  Copies both to the host and runs
 * the traversal there (O(m + nnz)), then writes the lists back; synchronises
 * `stream`.  SPMM_ERR_INVALID_CSR if row_ptr does not start at 0 or
 * decreases.  The pages have no row reordering; this extends the plan's
 * analysis reuse. */
spmm_status_t spmm_plan_order_rows(spmm_plan_t plan, const int32_t *row_ptr,
                                   const int32_t *col_idx, void *stream);

/* The same reorder, kept only where it raises B-row reuse: over windows of 64
 * consecutive list rows (about the rows one SM has in flight), the distinct
 * B rows per stored entry must fall by at least a tenth in breadth-first
 * order.  Otherwise (uniformly random columns, where the reorder only
 * scatters the rows, or a numbering that is already local, like a row-major
 * stencil) the lists are left as they are.  *applied (required) is set to 1
 * when the order was changed, else 0.  Same arguments, errors and
 * synchronisation as spmm_plan_order_rows; the reuse count adds O(nnz + k)
 * host work. */
spmm_status_t spmm_plan_order_rows_auto(spmm_plan_t plan, const int32_t *row_ptr,
                                        const int32_t *col_idx, void *stream,
                                        int32_t *applied);

/* Host function (no GPU involved): order[i] = the i-th row of an m-row CSR
 * pattern (HOST arrays row_ptr[m + 1], col_idx[row_ptr[m]]) in breadth-first
 * order.  Row i is adjacent to row j for each stored entry (i, j) with
 * 0 <= j < m; other columns are skipped.  The traversal starts at row 0,
 * visits each row's neighbours in stored order, and restarts at the lowest
 * unvisited row when a component is exhausted, so `order` (caller-owned, m
 * entries) is a permutation of 0..m-1.  SPMM_ERR_INVALID_CSR if row_ptr[0] != 0
 * or row_ptr decreases; SPMM_ERR_NULL_POINTER for a missing array (col_idx
 * may be NULL when the pattern is empty). */
spmm_status_t spmm_row_order_bfs(const int32_t *row_ptr, const int32_t *col_idx, int64_t m,
                                 int32_t *order);

/* C = alpha * A * B + beta * C with A's structure taken from the plan.
 * row_ptr must hold the structure the plan analysed (same values); col_idx,
 * values, B and C may change from call to call.  Same argument rules as
 * spmm_csr_f32 (m, k, n come from the plan).  SPMM_ERR_INVALID_ARGUMENT if the
 * plan was made for the other element size.  Asynchronous on `stream`. */
spmm_status_t spmm_plan_csr_f32(spmm_plan_t plan, float alpha,
                                const int32_t *row_ptr, const int32_t *col_idx,
                                const float *values, const float *B, int64_t ldb,
                                float beta, float *C, int64_t ldc, void *stream);

/* Same in binary64. */
spmm_status_t spmm_plan_csr_f64(spmm_plan_t plan, double alpha,
                                const int32_t *row_ptr, const int32_t *col_idx,
                                const double *values, const double *B, int64_t ldb,
                                double beta, double *C, int64_t ldc, void *stream);

/* Per-stage record of the most recent product issued on a handle with
 * profiling enabled (a tracing aid; the pages have no counterpart).  Times are
 * GPU durations between CUDA events recorded on the call's stream around each
 * stage; the counts come from the device-side row bins. */
typedef struct {
    float prepass_ms;      /* row-binning pre-pass (1 to 3 launches; none for m <= 2048,
                              where the whole product is one launch: rows_ms) */
    float rows_ms;         /* short + medium rows kernel (1 launch) */
    float long_ms;         /* long-row CTA split (1 launch) */
    float fixup_ms;        /* 0: the long-row fixup runs inside the long-row launch */
    float total_ms;        /* first event to last event */
    int32_t launches;      /* kernels the product launched */
    int32_t rows_short, rows_medium, rows_long;  /* rows per bin */
    int32_t long_nnz;      /* entries in long rows */
    int32_t panels, panel_cols;                  /* column panels of B/C */
    int32_t vec_elems, group_lanes, slots;       /* kernel geometry: W, G, R */
    int32_t short_max, long_min;                 /* bin thresholds (row lengths) */
} spmm_profile_t;

/* Turn per-stage event recording on (enable != 0) or off for later calls on
 * this handle.  Off by default; recording adds a few events per call. */
spmm_status_t spmm_set_profiling(spmm_handle_t h, int enable);

/* Read the record of the most recent profiled product (waits for its events
 * and copies the bin counts to the host).  SPMM_ERR_INVALID_ARGUMENT if no
 * profiled product has been issued.  Only the epilogue-only path ran when
 * launches == 1 and rows_ms == 0. */
spmm_status_t spmm_get_profile(spmm_handle_t h, spmm_profile_t *out);

/* Measurement aid (the pages have no counterpart): the device's binary64
 * fused multiply-add rate, against which binary64 products are measured on
 * parts whose FP64 units, not memory, bound them.  Runs a kernel in which
 * every thread advances eight independent chains of fma.rn.f64 (32 warps per
 * SM), times three launches after a warm-up with CUDA events on the legacy
 * default stream, and writes the best rate in FMA instructions per second
 * (one FMA = 2 flops) to *fma_per_second.  Synchronises the device; uses 8
 * bytes of handle scratch per thread (1024 threads per SM). */
spmm_status_t spmm_measure_fp64_fma_rate(spmm_handle_t h, double *fma_per_second);

/* C = alpha * A * B + beta * C in binary32 without allocating anything.
 *
 * For callers that cannot call cudaMalloc: code running under a fixed or
 * capped memory budget, inside an allocator or a host framework that owns all
 * device memory, or on a path that must never stall on an allocation.  The
 * reference pages have no counterpart; this is an addition of this library.
 *
 * Same operation, conventions, arguments (minus the handle) and results as
 * spmm_csr_f32, on the same kernels.  The scratch they need (row bins, long-row
 * partial sums) is one fixed device array inside the library, about 11 MB,
 * held by every GPU that loads the library until the process exits.  Limits:
 * m <= 524288 and n <= 512; larger products return SPMM_ERR_TOO_LARGE and do
 * nothing.  The call never calls cudaMalloc, cudaFree or any allocating
 * routine.
 *
 * The first call on a device (with that device current) looks up the array's
 * device address and the device's SM count and L2 size; make that first call
 * before capturing any stream into a CUDA graph.  Every call on a device shares
 * the one array, which keeps the last call's contents: calls whose work
 * overlaps on the GPU (different streams, or different host threads) race and
 * must be serialised by the caller.  Nothing in the array needs to start at
 * zero.  Asynchronous on `stream`, like spmm_csr_f32.  The array's address
 * is looked up once per device and kept: after cudaDeviceReset on a device
 * the address may no longer be valid, so the entry point must not be called
 * on that device again in the same process.  A device with more than 160
 * SMs (more long-row CTAs than the array holds partial sums for) gets
 * SPMM_ERR_UNSUPPORTED_DEVICE. */
spmm_status_t spmm_csr_f32_noalloc(float alpha,
                                   const int32_t *row_ptr, const int32_t *col_idx,
                                   const float *values, int64_t m, int64_t k,
                                   const float *B, int64_t ldb, int64_t n,
                                   float beta, float *C, int64_t ldc, void *stream);

/* Static, human-readable name of a status code (never NULL). */
const char *spmm_status_string(spmm_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* CSR_SPMM_H */
