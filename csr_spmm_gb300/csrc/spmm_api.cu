// Host driver behind the C ABI in include/csr_spmm.h: argument validation,
// the handle and its scratch, the column-panel / geometry plan, and the
// launch sequence
//   pre-pass (row bins) -> short/medium rows -> long-row CTA split (+ fixup).
// No step synchronises the stream; no device value is read back.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "csr_spmm.h"
#include "spmm_internal.h"
#include "spmm_ops.h"

using namespace spmm;

struct spmm_handle_s {
    int device = 0;
    int num_sms = 0;
    int64_t l2_bytes = 0;
    int64_t persist_max = 0;          // largest persisting L2 set-aside
    int64_t window_max = 0;           // largest access-policy window
    int64_t persist_bytes = 0;        // set-aside this handle asked for (0: off)
    size_t persist_prev = 0;          // the limit before, restored on destroy
    void* scratch = nullptr;
    size_t scratch_bytes = 0;
    int* check_status = nullptr;
    // occupancy cache of the rows kernel, keyed by (element size, W, G, R)
    struct OccEntry { int es, W, G, R, blocks; };
    OccEntry occ[32];
    int nocc = 0;
    // profiling: events around the stages of the last profiled call
    bool profiling = false;
    bool have_profile = false;
    cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
    spmm_profile_t prof{};
    const int* prof_hdr = nullptr;     // device header of the last profiled call
};

// An analysed sparsity structure: the row bins of one row_ptr, computed once
// and reused by every product issued on the plan.
struct spmm_plan_s {
    spmm_handle_s* h = nullptr;
    int device = 0;                   // the handle's device (destroy needs no handle)
    int64_t m = 0, k = 0, n = 0;
    int es = 0;
    int long_grid = 0;
    void* scratch = nullptr;          // bins, counters, partials (plan-owned)
    int* hdr = nullptr;
    int* rowlist = nullptr;
    int* med_pre = nullptr;
    int* long_pre = nullptr;
    int* long_cnt = nullptr;
    void* partials = nullptr;
    int hdr_host[HDR_WORDS] = {};     // bin counts, read back once
};

namespace spmm {

// Fraction of L2 a B column panel may occupy; panels are only used when B
// itself exceeds PANEL_TRIGGER of L2.
#ifndef SPMM_PANEL_FRACTION
#define SPMM_PANEL_FRACTION 0.5
#endif
#ifndef SPMM_PANEL_TRIGGER
#define SPMM_PANEL_TRIGGER 3.0
#endif
#ifndef SPMM_PANEL_COLS
#define SPMM_PANEL_COLS 0     // > 0 forces the panel width (tuning experiments)
#endif
constexpr double PANEL_FRACTION = SPMM_PANEL_FRACTION;
constexpr double PANEL_TRIGGER = SPMM_PANEL_TRIGGER;
// Rows at least this long go to the CTA-split kernel.
#ifndef SPMM_LONG_MIN_ROW
#define SPMM_LONG_MIN_ROW 1024
#endif
constexpr int LONG_MIN_ROW = SPMM_LONG_MIN_ROW;
// Narrow lane groups: rows of up to this many group steps stay in the short
// bin (one group per row); longer ones get a whole warp (medium bin).
#ifndef SPMM_SHORT_MAX_STEPS
#define SPMM_SHORT_MAX_STEPS 2
#endif
// Long-row grid: CTAs per SM.
#ifndef SPMM_LONG_CTAS
#define SPMM_LONG_CTAS 4
#endif
constexpr int LONG_CTAS_PER_SM = SPMM_LONG_CTAS;

int long_grid_for(int num_sms) { return LONG_CTAS_PER_SM * num_sms; }

// Geometry for a product with k x n B of element size es on a device with
// l2_bytes of L2; `vec` when B and C allow 16-byte accesses (base pointers
// and leading dimensions).
ProductPlan plan_product(int64_t l2_bytes, int64_t k, int64_t n, int es, bool vec) {
    const int WV = 16 / es;
    ProductPlan P{};
    P.geo.W = vec ? WV : 1;
    const int W = P.geo.W;

    // column panels: keep the B panel being gathered resident in L2
    int64_t panel = n;
    const double bbytes = (double)k * (double)n * es;
    if (l2_bytes > 0 && bbytes > PANEL_TRIGGER * (double)l2_bytes) {
        const int64_t align = std::max<int64_t>(W, 128 / es);      // whole 128-byte lines
        int64_t cols = (int64_t)(PANEL_FRACTION * (double)l2_bytes / ((double)k * es));
        cols = cols / align * align;
        if (cols < align) cols = std::max<int64_t>(W, align);
        const int64_t np = (n + cols - 1) / cols;
        panel = (n + np - 1) / np;
        panel = (panel + W - 1) / W * W;
    }
    if (SPMM_PANEL_COLS > 0) panel = (SPMM_PANEL_COLS + W - 1) / W * W;
    P.panel_cols = (int)std::min<int64_t>(panel, n);
    P.npanels = (int)((n + P.panel_cols - 1) / P.panel_cols);

    const int nvec = (P.panel_cols + W - 1) / W;
    if (nvec <= 32) {
        int g = 1;
        while (g < nvec) g <<= 1;
        P.geo.G = g;
        P.geo.R = 1;
    } else {
        P.geo.G = 32;
        P.geo.R = nvec <= 64 ? 2 : 4;
    }
    P.geo.whole = (n % W) == 0;
    // Bin thresholds: those of the 16-byte geometry whatever the operands'
    // alignment, so that the bins, and with them the summation order of every
    // row, depend only on the row lengths, n and the element size.  A plan
    // (binned once, for 16-byte operands) then gives the direct call's
    // results bit for bit for any alignment; any threshold is correct for
    // every geometry.
    if (!vec) {
        const ProductPlan V = plan_product(l2_bytes, k, n, es, true);
        P.short_max = V.short_max;
        P.long_min = V.long_min;
        return P;
    }
    const int bytes_per_entry = P.geo.R * W * es;
    const int batch_bytes = es == 8 ? SPMM_BATCH_BYTES_F64 : SPMM_BATCH_BYTES;
    const int U = std::min(SPMM_BATCH_MAX, std::max(1, batch_bytes / bytes_per_entry));
    const int CH = std::max(P.geo.G, U);
    P.long_min = LONG_MIN_ROW;
    P.short_max = (P.geo.G == 32) ? P.long_min - 1
                                  : std::min(P.long_min - 1, SPMM_SHORT_MAX_STEPS * CH);
    return P;
}

}  // namespace spmm

namespace {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

struct ScratchLayout {
    size_t hdr, tile_counts, tile_offsets, rowlist, med_pre, long_pre, long_cnt, partials, total;
};

ScratchLayout layout_for(int64_t m, int64_t n, int es, int long_grid) {
    ScratchLayout L{};
    const int64_t tiles = (m + BIN_TILE - 1) / BIN_TILE;
    size_t off = 0;
    L.hdr = off;          off = align_up(off + sizeof(int) * HDR_WORDS, 256);
    L.tile_counts = off;  off = align_up(off + sizeof(int) * BIN_REC * (size_t)std::max<int64_t>(tiles, 1), 256);
    L.tile_offsets = off; off = align_up(off + sizeof(int) * BIN_REC * (size_t)std::max<int64_t>(tiles, 1), 256);
    L.rowlist = off;      off = align_up(off + sizeof(int) * (size_t)std::max<int64_t>(m, 1), 256);
    L.med_pre = off;      off = align_up(off + sizeof(int) * (size_t)(m + 1), 256);
    L.long_pre = off;     off = align_up(off + sizeof(int) * (size_t)(m + 1), 256);
    L.long_cnt = off;     off = align_up(off + sizeof(int) * (size_t)std::max<int64_t>(m, 1), 256);
    L.partials = off;     off = align_up(off + (size_t)es * 2 * long_grid * (size_t)std::max<int64_t>(n, 1), 256);
    L.total = off;
    return L;
}

int long_grid_of(const spmm_handle_s* h) { return long_grid_for(h->num_sms); }

spmm_status_t ensure_scratch(spmm_handle_s* h, size_t bytes) {
    if (bytes <= h->scratch_bytes) return SPMM_OK;
    if (h->scratch) {
        cudaDeviceSynchronize();     // earlier calls may still use the old buffer
        cudaFree(h->scratch);
        h->scratch = nullptr;
        h->scratch_bytes = 0;
    }
    const size_t want = align_up(bytes + bytes / 4, 1 << 20);
    if (cudaMalloc(&h->scratch, want) != cudaSuccess) {
        cudaGetLastError();
        h->scratch = nullptr;
        return SPMM_ERR_ALLOC;
    }
    h->scratch_bytes = want;
    return SPMM_OK;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

using Plan = ProductPlan;

Plan make_plan_es(const spmm_handle_s* h, int64_t k, int64_t n, int es, bool vec) {
    return plan_product(h->l2_bytes, k, n, es, vec);
}

template <typename T>
Plan make_plan(const spmm_handle_s* h, int64_t k, int64_t n, const T* B, int64_t ldb, const T* C,
               int64_t ldc) {
    const int WV = 16 / (int)sizeof(T);
    const bool vec = aligned(B, 16) && aligned(C, 16) && ldb % WV == 0 && ldc % WV == 0;
    return make_plan_es(h, k, n, (int)sizeof(T), vec);
}

// Access-policy window over the B rows a product gathers, when the handle
// holds a persisting L2 set-aside and B's span fits in it: B's lines then
// persist, and the A and C streams cannot evict them.  A B larger than the
// set-aside gets no window (measured on GB300: persisting a fraction of a
// larger B slowed the product by 5-10%).
template <typename T>
const L2Window* b_window(const spmm_handle_s* h, const T* B, int64_t k, int64_t ldb, int64_t n,
                         L2Window* w) {
    if (h->persist_bytes <= 0 || k <= 0 || n <= 0) return nullptr;
    const double span = ((double)(k - 1) * (double)ldb + (double)n) * sizeof(T);
    if (span > (double)h->persist_bytes || span > (double)h->window_max) return nullptr;
    w->base = B;
    w->bytes = (size_t)span;
    w->hit_ratio = 1.0f;
    return w;
}

int rows_grid(spmm_handle_s* h, int es, const Geometry& g) {
    for (int i = 0; i < h->nocc; ++i) {
        const auto& e = h->occ[i];
        if (e.es == es && e.W == g.W && e.G == g.G && e.R == g.R) return e.blocks * h->num_sms;
    }
    const int b = es == 4 ? rows_blocks_per_sm<float>(g) : rows_blocks_per_sm<double>(g);
    if (h->nocc < 32) h->occ[h->nocc++] = {es, g.W, g.G, g.R, b};
    return b * h->num_sms;
}

// m <= SMALL_ROWS: the whole product in one launch, no pre-pass and no
// handle scratch.  Profiling counts every row as short (the kernel bins them
// itself) and reports the one launch as the rows stage.
template <typename T>
spmm_status_t small_product(spmm_handle_s* h, const Plan& P, const SpmmParams<T>& p,
                            const L2Window* win, cudaStream_t st);

// Records event i of the profiled call (no-op when profiling is off).
inline void mark(spmm_handle_s* h, int i, cudaStream_t st) {
    if (h->profiling) cudaEventRecord(h->ev[i], st);
}

template <typename T>
spmm_status_t small_product(spmm_handle_s* h, const Plan& P, const SpmmParams<T>& p,
                            const L2Window* win, cudaStream_t st) {
    mark(h, 0, st);
    mark(h, 1, st);
    if (launch_small<T>(p, P.geo, P.short_max, h->num_sms, st, win) != cudaSuccess)
        return SPMM_ERR_CUDA;
    mark(h, 2, st);
    mark(h, 3, st);
    mark(h, 4, st);
    if (h->profiling) {
        h->prof = spmm_profile_t{};
        h->prof.launches = 1;
        h->prof.rows_short = p.m;
        h->prof.panels = P.npanels;
        h->prof.panel_cols = P.panel_cols;
        h->prof.vec_elems = P.geo.W;
        h->prof.group_lanes = P.geo.G;
        h->prof.slots = P.geo.R;
        h->prof.short_max = P.short_max;
        h->prof.long_min = P.long_min;
        h->prof_hdr = nullptr;
        h->have_profile = true;
    }
    return SPMM_OK;
}

template <typename T>
spmm_status_t spmm_csr_impl(spmm_handle_t h, T alpha, const int32_t* row_ptr,
                            const int32_t* col_idx, const T* values, int64_t m, int64_t k,
                            const T* B, int64_t ldb, int64_t n, T beta, T* C, int64_t ldc,
                            void* stream) {
    // ---- validation (oxicuda-sparse, ops/spmm.rs, `spmm`: dimension checks) ----
    if (!h) return SPMM_ERR_INVALID_ARGUMENT;
    if (m < 0 || k < 0 || n < 0) return SPMM_ERR_INVALID_ARGUMENT;
    if (m > (int64_t)INT_MAX - BIN_TILE || k > (int64_t)INT_MAX || n > (int64_t)INT_MAX)
        return SPMM_ERR_INVALID_ARGUMENT;
    if (ldb < std::max<int64_t>(1, n) || ldc < std::max<int64_t>(1, n))
        return SPMM_ERR_DIMENSION_MISMATCH;
    if (ldb > (int64_t)INT_MAX) return SPMM_ERR_INVALID_ARGUMENT;   // 32-bit gather offsets
    if (m == 0 || n == 0) return SPMM_OK;             // nothing to compute (as on the page)
    if (!C) return SPMM_ERR_NULL_POINTER;
    const bool uses_a = alpha != T(0) && k > 0;
    if (uses_a && (!row_ptr || !col_idx || !values || !B)) return SPMM_ERR_NULL_POINTER;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    if (!uses_a) {
        // alpha == 0 or k == 0: C = beta * C, A and B not read
        const int grid = h->num_sms * 8;
        if (h->profiling) {
            h->prof = spmm_profile_t{};
            h->prof.launches = 1;
            h->prof_hdr = nullptr;
            for (int i = 0; i < 5; ++i) mark(h, i, st);
            h->have_profile = true;
        }
        return launch_scale<T>(C, ldc, (int)m, (int)n, beta, grid, st) == cudaSuccess
                   ? SPMM_OK : SPMM_ERR_CUDA;
    }

    const Plan P = make_plan<T>(h, k, n, B, ldb, C, ldc);
    if (m <= SMALL_ROWS) {
        SpmmParams<T> p{};
        p.row_ptr = row_ptr;
        p.col_idx = col_idx;
        p.values = values;
        p.B = B;
        p.ldb = ldb;
        p.C = C;
        p.ldc = ldc;
        p.m = (int)m;
        p.n = (int)n;
        p.alpha = alpha;
        p.beta = beta;
        p.panel_cols = P.panel_cols;
        p.npanels = P.npanels;
        L2Window wbuf;
        return small_product<T>(h, P, p, b_window(h, B, k, ldb, n, &wbuf), st);
    }
    const int lg = long_grid_of(h);
    const ScratchLayout L = layout_for(m, n, (int)sizeof(T), lg);
    spmm_status_t s = ensure_scratch(h, L.total);
    if (s != SPMM_OK) return s;
    char* base = static_cast<char*>(h->scratch);

    BinScratch bs{};
    bs.hdr = reinterpret_cast<int*>(base + L.hdr);
    bs.tile_counts = reinterpret_cast<int*>(base + L.tile_counts);
    bs.tile_offsets = reinterpret_cast<int*>(base + L.tile_offsets);
    bs.rowlist = reinterpret_cast<int*>(base + L.rowlist);
    bs.med_pre = reinterpret_cast<int*>(base + L.med_pre);
    bs.long_pre = reinterpret_cast<int*>(base + L.long_pre);
    bs.long_cnt = reinterpret_cast<int*>(base + L.long_cnt);
    bin_geometry(m, &bs.items, &bs.tiles);

    // overlap launches only when no profiling events sit between the kernels
    const bool overlap = SPMM_PDL && !h->profiling;
    mark(h, 0, st);
    if (launch_binning(row_ptr, (int)m, P.short_max, P.long_min, bs, st, overlap) != cudaSuccess)
        return SPMM_ERR_CUDA;
    mark(h, 1, st);

    SpmmParams<T> p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.values = values;
    p.B = B;
    p.ldb = ldb;
    p.C = C;
    p.ldc = ldc;
    p.m = (int)m;
    p.n = (int)n;
    p.alpha = alpha;
    p.beta = beta;
    p.panel_cols = P.panel_cols;
    p.npanels = P.npanels;
    p.rowlist = bs.rowlist;
    p.med_pre = bs.med_pre;
    p.long_pre = bs.long_pre;
    p.long_cnt = bs.long_cnt;
    p.hdr = bs.hdr;
    p.partials = reinterpret_cast<T*>(base + L.partials);
    p.long_grid = lg;

    L2Window wbuf;
    const L2Window* win = b_window(h, B, k, ldb, n, &wbuf);
    if (launch_rows<T>(p, P.geo, rows_grid(h, (int)sizeof(T), P.geo), st, overlap, win) !=
        cudaSuccess)
        return SPMM_ERR_CUDA;
    mark(h, 2, st);
    if (launch_long<T>(p, P.geo, st, overlap, win) != cudaSuccess) return SPMM_ERR_CUDA;
    mark(h, 3, st);
    mark(h, 4, st);               // the fixup runs inside the long-row launch
    if (h->profiling) {
        h->prof = spmm_profile_t{};
        h->prof.launches = binning_launches(m) + 2;
        h->prof.panels = P.npanels;
        h->prof.panel_cols = P.panel_cols;
        h->prof.vec_elems = P.geo.W;
        h->prof.group_lanes = P.geo.G;
        h->prof.slots = P.geo.R;
        h->prof.short_max = P.short_max;
        h->prof.long_min = P.long_min;
        h->prof_hdr = bs.hdr;
        h->have_profile = true;
    }
    return SPMM_OK;
}

template <typename T>
spmm_status_t spmm_plan_impl(spmm_plan_t pl, T alpha, const int32_t* row_ptr,
                             const int32_t* col_idx, const T* values, const T* B, int64_t ldb,
                             T beta, T* C, int64_t ldc, void* stream) {
    if (!pl || pl->es != (int)sizeof(T)) return SPMM_ERR_INVALID_ARGUMENT;
    spmm_handle_s* h = pl->h;
    const int64_t m = pl->m, k = pl->k, n = pl->n;
    if (ldb < std::max<int64_t>(1, n) || ldc < std::max<int64_t>(1, n))
        return SPMM_ERR_DIMENSION_MISMATCH;
    if (ldb > (int64_t)INT_MAX) return SPMM_ERR_INVALID_ARGUMENT;   // 32-bit gather offsets
    if (m == 0 || n == 0) return SPMM_OK;
    if (!C) return SPMM_ERR_NULL_POINTER;
    const bool uses_a = alpha != T(0) && k > 0;
    if (uses_a && (!row_ptr || !col_idx || !values || !B)) return SPMM_ERR_NULL_POINTER;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!uses_a) {
        if (h->profiling) {
            h->prof = spmm_profile_t{};
            h->prof.launches = 1;
            h->prof_hdr = nullptr;
            for (int i = 0; i < 5; ++i) mark(h, i, st);
            h->have_profile = true;
        }
        return launch_scale<T>(C, ldc, (int)m, (int)n, beta, h->num_sms * 8, st) == cudaSuccess
                   ? SPMM_OK : SPMM_ERR_CUDA;
    }
    const Plan P = make_plan<T>(h, k, n, B, ldb, C, ldc);
    SpmmParams<T> p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.values = values;
    p.B = B;
    p.ldb = ldb;
    p.C = C;
    p.ldc = ldc;
    p.m = (int)m;
    p.n = (int)n;
    p.alpha = alpha;
    p.beta = beta;
    p.panel_cols = P.panel_cols;
    p.npanels = P.npanels;
    p.rowlist = pl->rowlist;
    p.med_pre = pl->med_pre;
    p.long_pre = pl->long_pre;
    p.long_cnt = pl->long_cnt;
    p.hdr = pl->hdr;
    p.partials = static_cast<T*>(pl->partials);
    p.long_grid = pl->long_grid;
    if (m <= SMALL_ROWS) {                // the direct call's one-launch path, same bits
        L2Window wbuf;
        return small_product<T>(h, P, p, b_window(h, B, k, ldb, n, &wbuf), st);
    }
    const bool overlap = SPMM_PDL && !h->profiling;
    const bool has_long = pl->hdr_host[HDR_COUNT_LONG] > 0;
    mark(h, 0, st);
    mark(h, 1, st);                       // no pre-pass: the plan holds the bins
    // the first kernel of the call waits for the stream (no launch overlap)
    L2Window wbuf;
    const L2Window* win = b_window(h, B, k, ldb, n, &wbuf);
    if (launch_rows<T>(p, P.geo, rows_grid(h, (int)sizeof(T), P.geo), st, false, win) !=
        cudaSuccess)
        return SPMM_ERR_CUDA;
    mark(h, 2, st);
    if (has_long && launch_long<T>(p, P.geo, st, overlap, win) != cudaSuccess)
        return SPMM_ERR_CUDA;
    mark(h, 3, st);
    mark(h, 4, st);
    if (h->profiling) {
        h->prof = spmm_profile_t{};
        h->prof.launches = has_long ? 2 : 1;
        h->prof.panels = P.npanels;
        h->prof.panel_cols = P.panel_cols;
        h->prof.vec_elems = P.geo.W;
        h->prof.group_lanes = P.geo.G;
        h->prof.slots = P.geo.R;
        h->prof.short_max = P.short_max;
        h->prof.long_min = P.long_min;
        h->prof_hdr = pl->hdr;
        h->have_profile = true;
    }
    return SPMM_OK;
}

// The squared chain C = alpha * A (A B) + beta * C for a square A: the K^2 B
// product that the SEACells Frank-Wolfe kernels of the bixverse page consume
// (module doc: the n x k output of `k_squared_matmul`).  One pre-pass bins
// the rows for both products.  The intermediate T = A B lives in handle
// scratch with a 16-byte-aligned leading dimension and is stored with the
// default L2 policy (not streamed), so that the second product's gathers of
// T find it in L2 when it fits there.
// The two products of the squared chain on bins already made (p carries A,
// the bins and the partial-sum scratch): T = A B into Tm (leading dimension
// ldt, default L2 policy so the second product finds it), then C = alpha A T
// + beta C.  run_long: launch the long-row kernel (a plan knows whether its
// structure has long rows); first_overlap: the first launch may overlap its
// predecessor (the library's own pre-pass).  Marks profile events 2 and 3-4.
template <typename T>
spmm_status_t chain_products(spmm_handle_s* h, SpmmParams<T> p, const T* B, int64_t ldb, T* Tm,
                             int64_t ldt, T alpha, T beta, T* C, int64_t ldc, bool run_long,
                             bool first_overlap, bool overlap, cudaStream_t st) {
    const int64_t m = p.m, n = p.n;
    const Plan P1 = make_plan<T>(h, m, n, B, ldb, Tm, ldt);
    const Plan P2 = make_plan<T>(h, m, n, Tm, ldt, C, ldc);
    p.B = B;
    p.ldb = ldb;
    p.C = Tm;
    p.ldc = ldt;
    p.alpha = T(1);
    p.beta = T(0);
    p.keep_c = 1;
    p.panel_cols = P1.panel_cols;
    p.npanels = P1.npanels;
    L2Window w1;
    const L2Window* win1 = b_window(h, B, m, ldb, n, &w1);
    if (launch_rows<T>(p, P1.geo, rows_grid(h, (int)sizeof(T), P1.geo), st, first_overlap,
                       win1) != cudaSuccess ||
        (run_long && launch_long<T>(p, P1.geo, st, overlap, win1) != cudaSuccess))
        return SPMM_ERR_CUDA;
    mark(h, 2, st);
    p.B = Tm;
    p.ldb = ldt;
    p.C = C;
    p.ldc = ldc;
    p.alpha = alpha;
    p.beta = beta;
    p.keep_c = 0;
    p.panel_cols = P2.panel_cols;
    p.npanels = P2.npanels;
    L2Window w2;
    const L2Window* win2 = b_window(h, static_cast<const T*>(Tm), m, ldt, n, &w2);
    if (launch_rows<T>(p, P2.geo, rows_grid(h, (int)sizeof(T), P2.geo), st, overlap, win2) !=
            cudaSuccess ||
        (run_long && launch_long<T>(p, P2.geo, st, overlap, win2) != cudaSuccess))
        return SPMM_ERR_CUDA;
    mark(h, 3, st);
    mark(h, 4, st);
    return SPMM_OK;
}

template <typename T>
spmm_status_t spmm_squared_impl(spmm_handle_t h, T alpha, const int32_t* row_ptr,
                                const int32_t* col_idx, const T* values, int64_t m, const T* B,
                                int64_t ldb, int64_t n, T beta, T* C, int64_t ldc, void* stream) {
    if (!h) return SPMM_ERR_INVALID_ARGUMENT;
    if (m < 0 || n < 0) return SPMM_ERR_INVALID_ARGUMENT;
    if (m > (int64_t)INT_MAX - BIN_TILE || n > (int64_t)INT_MAX) return SPMM_ERR_INVALID_ARGUMENT;
    if (ldb < std::max<int64_t>(1, n) || ldc < std::max<int64_t>(1, n))
        return SPMM_ERR_DIMENSION_MISMATCH;
    if (ldb > (int64_t)INT_MAX) return SPMM_ERR_INVALID_ARGUMENT;
    if (m == 0 || n == 0) return SPMM_OK;
    if (!C) return SPMM_ERR_NULL_POINTER;
    const bool uses_a = alpha != T(0);
    if (uses_a && (!row_ptr || !col_idx || !values || !B)) return SPMM_ERR_NULL_POINTER;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!uses_a) {
        if (h->profiling) {
            h->prof = spmm_profile_t{};
            h->prof.launches = 1;
            h->prof_hdr = nullptr;
            for (int i = 0; i < 5; ++i) mark(h, i, st);
            h->have_profile = true;
        }
        return launch_scale<T>(C, ldc, (int)m, (int)n, beta, h->num_sms * 8, st) == cudaSuccess
                   ? SPMM_OK : SPMM_ERR_CUDA;
    }

    constexpr int64_t WV = 16 / (int64_t)sizeof(T);
    const int64_t ldt = (n + WV - 1) / WV * WV;
    if (ldt > (int64_t)INT_MAX) return SPMM_ERR_INVALID_ARGUMENT;
    const int lg = long_grid_of(h);
    const ScratchLayout L = layout_for(m, n, (int)sizeof(T), lg);
    const size_t t_off = align_up(L.total, 256);
    spmm_status_t s = ensure_scratch(h, t_off + (size_t)m * (size_t)ldt * sizeof(T));
    if (s != SPMM_OK) return s;
    char* base = static_cast<char*>(h->scratch);
    T* Tm = reinterpret_cast<T*>(base + t_off);

    BinScratch bs{};
    bs.hdr = reinterpret_cast<int*>(base + L.hdr);
    bs.tile_counts = reinterpret_cast<int*>(base + L.tile_counts);
    bs.tile_offsets = reinterpret_cast<int*>(base + L.tile_offsets);
    bs.rowlist = reinterpret_cast<int*>(base + L.rowlist);
    bs.med_pre = reinterpret_cast<int*>(base + L.med_pre);
    bs.long_pre = reinterpret_cast<int*>(base + L.long_pre);
    bs.long_cnt = reinterpret_cast<int*>(base + L.long_cnt);
    bin_geometry(m, &bs.items, &bs.tiles);

    // first product T = A B; the bins it makes serve both products (they are
    // valid for any geometry)
    const Plan P1 = make_plan<T>(h, m, n, B, ldb, Tm, ldt);
    const bool overlap = SPMM_PDL && !h->profiling;
    mark(h, 0, st);
    if (launch_binning(row_ptr, (int)m, P1.short_max, P1.long_min, bs, st, overlap) != cudaSuccess)
        return SPMM_ERR_CUDA;
    mark(h, 1, st);

    SpmmParams<T> p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.values = values;
    p.m = (int)m;
    p.n = (int)n;
    p.rowlist = bs.rowlist;
    p.med_pre = bs.med_pre;
    p.long_pre = bs.long_pre;
    p.long_cnt = bs.long_cnt;
    p.hdr = bs.hdr;
    p.partials = reinterpret_cast<T*>(base + L.partials);
    p.long_grid = lg;
    s = chain_products<T>(h, p, B, ldb, Tm, ldt, alpha, beta, C, ldc, true, overlap, overlap, st);
    if (s != SPMM_OK) return s;
    if (h->profiling) {
        const Plan P2 = make_plan<T>(h, m, n, Tm, ldt, C, ldc);
        h->prof = spmm_profile_t{};
        h->prof.launches = binning_launches(m) + 4;
        h->prof.panels = P2.npanels;
        h->prof.panel_cols = P2.panel_cols;
        h->prof.vec_elems = P2.geo.W;
        h->prof.group_lanes = P2.geo.G;
        h->prof.slots = P2.geo.R;
        h->prof.short_max = P1.short_max;
        h->prof.long_min = P1.long_min;
        h->prof_hdr = bs.hdr;
        h->have_profile = true;
    }
    return SPMM_OK;
}

// The squared chain through a plan: the plan's bins (and row order) serve both
// products; the intermediate lives in the plan's handle's scratch.
template <typename T>
spmm_status_t spmm_plan_squared_impl(spmm_plan_t pl, T alpha, const int32_t* row_ptr,
                                     const int32_t* col_idx, const T* values, const T* B,
                                     int64_t ldb, T beta, T* C, int64_t ldc, void* stream) {
    if (!pl || pl->es != (int)sizeof(T) || pl->m != pl->k) return SPMM_ERR_INVALID_ARGUMENT;
    spmm_handle_s* h = pl->h;
    const int64_t m = pl->m, n = pl->n;
    if (ldb < std::max<int64_t>(1, n) || ldc < std::max<int64_t>(1, n))
        return SPMM_ERR_DIMENSION_MISMATCH;
    if (ldb > (int64_t)INT_MAX) return SPMM_ERR_INVALID_ARGUMENT;
    if (m == 0 || n == 0) return SPMM_OK;
    if (!C) return SPMM_ERR_NULL_POINTER;
    const bool uses_a = alpha != T(0);
    if (uses_a && (!row_ptr || !col_idx || !values || !B)) return SPMM_ERR_NULL_POINTER;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!uses_a) {
        if (h->profiling) {
            h->prof = spmm_profile_t{};
            h->prof.launches = 1;
            h->prof_hdr = nullptr;
            for (int i = 0; i < 5; ++i) mark(h, i, st);
            h->have_profile = true;
        }
        return launch_scale<T>(C, ldc, (int)m, (int)n, beta, h->num_sms * 8, st) == cudaSuccess
                   ? SPMM_OK : SPMM_ERR_CUDA;
    }
    constexpr int64_t WV = 16 / (int64_t)sizeof(T);
    const int64_t ldt = (n + WV - 1) / WV * WV;
    if (ldt > (int64_t)INT_MAX) return SPMM_ERR_INVALID_ARGUMENT;
    spmm_status_t s = ensure_scratch(h, (size_t)m * (size_t)ldt * sizeof(T));
    if (s != SPMM_OK) return s;
    T* Tm = static_cast<T*>(h->scratch);

    SpmmParams<T> p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.values = values;
    p.m = (int)m;
    p.n = (int)n;
    p.rowlist = pl->rowlist;
    p.med_pre = pl->med_pre;
    p.long_pre = pl->long_pre;
    p.long_cnt = pl->long_cnt;
    p.hdr = pl->hdr;
    p.partials = static_cast<T*>(pl->partials);
    p.long_grid = pl->long_grid;
    const bool overlap = SPMM_PDL && !h->profiling;
    mark(h, 0, st);
    mark(h, 1, st);                       // no pre-pass: the plan holds the bins
    s = chain_products<T>(h, p, B, ldb, Tm, ldt, alpha, beta, C, ldc,
                          pl->hdr_host[HDR_COUNT_LONG] > 0, false, overlap, st);
    if (s != SPMM_OK) return s;
    if (h->profiling) {
        const Plan P2 = make_plan<T>(h, m, n, Tm, ldt, C, ldc);
        h->prof = spmm_profile_t{};
        h->prof.launches = pl->hdr_host[HDR_COUNT_LONG] > 0 ? 4 : 2;
        h->prof.panels = P2.npanels;
        h->prof.panel_cols = P2.panel_cols;
        h->prof.vec_elems = P2.geo.W;
        h->prof.group_lanes = P2.geo.G;
        h->prof.slots = P2.geo.R;
        h->prof.short_max = P2.short_max;
        h->prof.long_min = P2.long_min;
        h->prof_hdr = pl->hdr;
        h->have_profile = true;
    }
    return SPMM_OK;
}

// The Frank-Wolfe gradient scan of the SEACells B update (bixverse page,
// seacells_kernels.rs, `fw_argmin_b` / `reduce_argmin_blocks`).
template <typename T>
spmm_status_t spmm_fw_impl(spmm_handle_t h, int64_t n, int64_t k, const int32_t* k2b_rp,
                           const int32_t* k2b_ci, const T* k2b_v, const int32_t* t1_rp,
                           const int32_t* t1_ci, const T* t1_v, const int32_t* t2_rp,
                           const int32_t* t2_ci, const T* t2_v, const int32_t* b_rp,
                           const int32_t* b_ci, const T* b_v, T* min_val, int32_t* min_idx,
                           T* gap, void* stream) {
    if (!h || n < 0 || k < 0) return SPMM_ERR_INVALID_ARGUMENT;
    constexpr int64_t TILE = fw_tile<T>();
    if (n > (int64_t)INT_MAX - 1 || k > (int64_t)INT_MAX / 2 - TILE) return SPMM_ERR_INVALID_ARGUMENT;
    if (!gap) return SPMM_ERR_NULL_POINTER;
    if (k > 0 && (!t1_rp || !t1_ci || !t1_v || !min_val || !min_idx)) return SPMM_ERR_NULL_POINTER;
    if (n > 0 && (!k2b_rp || !k2b_ci || !k2b_v || !t2_rp || !t2_ci || !t2_v || !b_rp || !b_ci ||
                  !b_v))
        return SPMM_ERR_NULL_POINTER;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t ldk = std::max<int64_t>(TILE, (k + TILE - 1) / TILE * TILE);
    const int grid = fw_blocks_per_sm<T>((int)k) * h->num_sms;
    const int nwarps = grid * (FW_THREADS / 32);
    size_t off = 0;
    const size_t o_t1 = off;   off = align_up(off + sizeof(T) * (size_t)k * ldk, 256);
    const size_t o_pv = off;   off = align_up(off + sizeof(T) * (size_t)grid * ldk, 256);
    const size_t o_pi = off;   off = align_up(off + sizeof(int) * (size_t)grid * ldk, 256);
    const size_t o_pg = off;   off = align_up(off + sizeof(double) * (size_t)grid, 256);
    spmm_status_t s = ensure_scratch(h, off);
    if (s != SPMM_OK) return s;
    char* base = static_cast<char*>(h->scratch);
    FwParams<T> p{};
    p.n = (int)n;
    p.k = (int)k;
    p.ldk = (int)ldk;
    p.k2b_rp = k2b_rp; p.k2b_ci = k2b_ci; p.k2b_v = k2b_v;
    p.t1_rp = t1_rp;   p.t1_ci = t1_ci;   p.t1_v = t1_v;
    p.t2_rp = t2_rp;   p.t2_ci = t2_ci;   p.t2_v = t2_v;
    p.b_rp = b_rp;     p.b_ci = b_ci;     p.b_v = b_v;
    p.t1d = reinterpret_cast<T*>(base + o_t1);
    p.part_val = reinterpret_cast<T*>(base + o_pv);
    p.part_idx = reinterpret_cast<int*>(base + o_pi);
    p.part_gap = reinterpret_cast<double*>(base + o_pg);
    p.nwarps = nwarps;
    p.nblocks = grid;
    p.out_val = min_val;
    p.out_idx = min_idx;
    p.out_gap = gap;
    return launch_fw<T>(p, grid, st) == cudaSuccess ? SPMM_OK : SPMM_ERR_CUDA;
}

// ILU(0) of the oxicuda preconditioner page, in place, scheduled on the
// device (dependency counts, then one persistent factorisation launch).
template <typename T>
spmm_status_t spmm_ilu0_impl(spmm_handle_t h, int64_t n, int64_t nnz, const int32_t* row_ptr,
                             const int32_t* col_idx, T* values, int32_t* depth, int32_t* status,
                             void* stream) {
    if (!h || n <= 0 || n > (int64_t)INT_MAX - 2 || nnz < 0 || nnz > (int64_t)INT_MAX)
        return SPMM_ERR_INVALID_ARGUMENT;
    if (!row_ptr || !col_idx || !values || !status) return SPMM_ERR_NULL_POINTER;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // int words: pending[n], cnt[n], head, tail, abort, finished | dep_ptr[n+1] | queue[n] |
    // dep_idx[nnz] | piv[nnz] (int2, 8-byte aligned) | rec[16 n] (int4, 16-byte aligned) |
    // pub[nnz] (T, 16-byte aligned) | done[n] | tile_sum[n / 1024]
    const size_t zero_words = 2 * (size_t)n + 4;
    const size_t o_ptr = zero_words, o_q = o_ptr + (size_t)n + 1, o_dep = o_q + (size_t)n;
    const size_t nz1 = (size_t)std::max<int64_t>(nnz, 1);
    const size_t o_piv = (o_dep + nz1 + 1) & ~(size_t)1;
    const size_t o_rec = (o_piv + 2 * nz1 + 3) & ~(size_t)3;          // 16-byte aligned
    const size_t o_pub = o_rec + 4 * (size_t)ILU0_REC_LANES * (size_t)n;
    const size_t o_done = o_pub + nz1 * (sizeof(T) / sizeof(int));
    const size_t o_tile = o_done + (size_t)n;
    const size_t words = o_tile + ((size_t)n + 1023) / 1024 + 1;
    spmm_status_t s = ensure_scratch(h, words * sizeof(int));
    if (s != SPMM_OK) return s;
    int* w = static_cast<int*>(h->scratch);
    if (cudaMemsetAsync(w, 0, zero_words * sizeof(int), st) != cudaSuccess ||
        cudaMemsetAsync(w + o_q, 0xff, (size_t)n * sizeof(int), st) != cudaSuccess ||
        cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) {
        cudaGetLastError();
        return SPMM_ERR_CUDA;
    }
    Ilu0Params<T> p{};
    p.n = (int)n;
    p.nnz = nnz;
    p.rp = row_ptr;
    p.ci = col_idx;
    p.v = values;
    p.depth = depth;
    p.pending = w;
    p.cnt = w + n;
    p.head = w + 2 * n;
    p.tail = w + 2 * n + 1;
    p.abort = w + 2 * n + 2;
    p.finished = w + 2 * n + 3;
    p.dep_ptr = w + o_ptr;
    p.queue = w + o_q;
    p.dep_idx = w + o_dep;
    p.piv = reinterpret_cast<int2*>(w + o_piv);
    p.rec = reinterpret_cast<int4*>(w + o_rec);
    p.tile_sum = w + o_tile;
    p.pub = reinterpret_cast<T*>(w + o_pub);
    p.done = w + o_done;
    p.status = status;
    const int grid = ilu0_blocks_per_sm<T>() * h->num_sms;
    return launch_ilu0<T>(p, grid, st) == cudaSuccess ? SPMM_OK : SPMM_ERR_CUDA;
}

// Distinct B rows gathered per entry, over windows of ROW_WINDOW consecutive
// rows of `rows` (the rows of one window run at about the same time on one
// SM, so a B row gathered twice within a window is likely an L1 hit).
// Columns outside [0, k) are not counted.
constexpr int ROW_WINDOW = 64;
double row_gather_spread(const int32_t* rp, const int32_t* ci, int64_t k,
                         const std::vector<int32_t>& rows) {
    std::vector<int32_t> stamp((size_t)std::max<int64_t>(k, 1), -1);
    int64_t distinct = 0, entries = 0;
    for (size_t i = 0; i < rows.size(); ++i) {
        const int32_t win = (int32_t)(i / ROW_WINDOW);
        const int32_t r = rows[i];
        for (int32_t q = rp[r]; q < rp[r + 1]; ++q) {
            const int32_t c = ci[q];
            if (c < 0 || c >= k) continue;
            ++entries;
            if (stamp[c] != win) {
                stamp[c] = win;
                ++distinct;
            }
        }
    }
    return entries > 0 ? (double)distinct / (double)entries : 1.0;
}

// Host part of spmm_plan_order_rows (may throw std::bad_alloc).
spmm_status_t plan_order_rows(spmm_plan_t pl, const int32_t* row_ptr, const int32_t* col_idx,
                              void* stream, bool automatic, int32_t* applied) {
    if (applied) *applied = 0;
    if (!pl) return SPMM_ERR_INVALID_ARGUMENT;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != pl->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    const int n_short = pl->hdr_host[HDR_COUNT_SHORT];
    const int n_med = pl->hdr_host[HDR_COUNT_MEDIUM];
    const int64_t m = pl->m;
    if (m == 0 || n_short + n_med == 0) return SPMM_OK;    // no rows binned: nothing to order
    if (!row_ptr) return SPMM_ERR_NULL_POINTER;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    auto fail = [] {
        cudaGetLastError();
        return SPMM_ERR_CUDA;
    };
    std::vector<int32_t> rp((size_t)m + 1);
    if (cudaMemcpyAsync(rp.data(), row_ptr, rp.size() * sizeof(int32_t), cudaMemcpyDeviceToHost,
                        st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return fail();
    if (!csr_rows_valid(rp.data(), m)) return SPMM_ERR_INVALID_CSR;
    const int64_t nnz = rp[m];
    if (nnz > 0 && !col_idx) return SPMM_ERR_NULL_POINTER;
    std::vector<int32_t> ci((size_t)nnz);
    std::vector<int32_t> list((size_t)n_short + n_med);
    if ((nnz > 0 && cudaMemcpyAsync(ci.data(), col_idx, ci.size() * sizeof(int32_t),
                                    cudaMemcpyDeviceToHost, st) != cudaSuccess) ||
        cudaMemcpyAsync(list.data(), pl->rowlist, list.size() * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return fail();
    std::vector<int32_t> order((size_t)m), rank((size_t)m);
    row_order_bfs(rp.data(), ci.data(), (int)m, order.data());
    for (int64_t i = 0; i < m; ++i) rank[order[i]] = (int32_t)i;
    auto by_rank = [&](int32_t a, int32_t b) { return rank[a] < rank[b]; };
    std::vector<int32_t> bfs(list);
    std::sort(bfs.begin(), bfs.begin() + n_short, by_rank);
    std::sort(bfs.begin() + n_short, bfs.end(), by_rank);
    // Keep the breadth-first order only where it makes neighbouring rows
    // gather the same B rows: the distinct B rows per window of consecutive
    // list rows (about the rows one SM has in flight) must fall by a tenth.
    // On uniformly random columns it does not, and reordering only scatters
    // the row accesses (measured slower there).
    if (automatic && !(row_gather_spread(rp.data(), ci.data(), pl->k, bfs) <=
                       0.9 * row_gather_spread(rp.data(), ci.data(), pl->k, list)))
        return SPMM_OK;
    list.swap(bfs);
    // prefix of medium-row lengths in the new list order (it balances medium
    // rows across warps by entries)
    std::vector<int32_t> med((size_t)n_med + 1, 0);
    for (int i = 0; i < n_med; ++i) {
        const int32_t r = list[(size_t)n_short + i];
        med[i + 1] = med[i] + (rp[r + 1] - rp[r]);
    }
    if (cudaMemcpyAsync(pl->rowlist, list.data(), list.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, st) != cudaSuccess ||
        (n_med > 0 && cudaMemcpyAsync(pl->med_pre, med.data(), med.size() * sizeof(int32_t),
                                      cudaMemcpyHostToDevice, st) != cudaSuccess) ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return fail();
    if (applied) *applied = 1;
    return SPMM_OK;
}

}  // namespace

extern "C" {

spmm_status_t spmm_create(spmm_handle_t* out, int device) {
    if (!out) return SPMM_ERR_NULL_POINTER;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess) {
        cudaGetLastError();
        return SPMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (device < 0 || device >= count) return SPMM_ERR_INVALID_ARGUMENT;
    int major = 0, minor = 0, sms = 0, l2 = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, device) != cudaSuccess) {
        cudaGetLastError();
        return SPMM_ERR_CUDA;
    }
    // the library carries sm_103a code only
    if (major != 10 || minor != 3) return SPMM_ERR_UNSUPPORTED_DEVICE;
    spmm_handle_s* h = new (std::nothrow) spmm_handle_s();
    if (!h) return SPMM_ERR_ALLOC;
    h->device = device;
    h->num_sms = sms;
    h->l2_bytes = l2;
    int pmax = 0, wmax = 0;
    if (cudaDeviceGetAttribute(&pmax, cudaDevAttrMaxPersistingL2CacheSize, device) == cudaSuccess &&
        cudaDeviceGetAttribute(&wmax, cudaDevAttrMaxAccessPolicyWindowSize, device) == cudaSuccess) {
        h->persist_max = pmax;
        h->window_max = wmax;
    }
    cudaGetLastError();
    *out = h;
    return SPMM_OK;
}

spmm_status_t spmm_destroy(spmm_handle_t h) {
    if (!h) return SPMM_OK;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != h->device) cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    for (auto& e : h->ev)
        if (e) cudaEventDestroy(e);
    if (h->scratch) cudaFree(h->scratch);
    if (h->check_status) cudaFree(h->check_status);
    if (h->persist_bytes > 0) {
        cudaCtxResetPersistingL2Cache();
        cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, h->persist_prev);
    }
    if (cur >= 0 && cur != h->device) cudaSetDevice(cur);
    cudaGetLastError();
    delete h;
    return SPMM_OK;
}

spmm_status_t spmm_reserve(spmm_handle_t h, int64_t m, int64_t n, int elem_size) {
    if (!h || m < 0 || n < 0 || (elem_size != 4 && elem_size != 8)) return SPMM_ERR_INVALID_ARGUMENT;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    return ensure_scratch(h, layout_for(m, n, elem_size, long_grid_of(h)).total);
}

spmm_status_t spmm_csr_f32(spmm_handle_t h, float alpha, const int32_t* row_ptr,
                           const int32_t* col_idx, const float* values, int64_t m, int64_t k,
                           const float* B, int64_t ldb, int64_t n, float beta, float* C,
                           int64_t ldc, void* stream) {
    return spmm_csr_impl<float>(h, alpha, row_ptr, col_idx, values, m, k, B, ldb, n, beta, C, ldc,
                                stream);
}

spmm_status_t spmm_csr_f64(spmm_handle_t h, double alpha, const int32_t* row_ptr,
                           const int32_t* col_idx, const double* values, int64_t m, int64_t k,
                           const double* B, int64_t ldb, int64_t n, double beta, double* C,
                           int64_t ldc, void* stream) {
    return spmm_csr_impl<double>(h, alpha, row_ptr, col_idx, values, m, k, B, ldb, n, beta, C,
                                 ldc, stream);
}

spmm_status_t spmm_csr_check(spmm_handle_t h, const int32_t* row_ptr, const int32_t* col_idx,
                             int64_t m, int64_t k, int64_t nnz, void* stream,
                             int32_t* host_status) {
    if (!h || !host_status) return !h ? SPMM_ERR_INVALID_ARGUMENT : SPMM_ERR_NULL_POINTER;
    if (m < 0 || k < 0 || nnz < 0) return SPMM_ERR_INVALID_ARGUMENT;
    if (!row_ptr || (nnz > 0 && !col_idx)) return SPMM_ERR_NULL_POINTER;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!h->check_status && cudaMalloc(&h->check_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        h->check_status = nullptr;
        return SPMM_ERR_ALLOC;
    }
    int status = 0;
    if (cudaMemsetAsync(h->check_status, 0, sizeof(int), st) != cudaSuccess ||
        launch_csr_check(row_ptr, col_idx, m, k, nnz, h->check_status, st) != cudaSuccess ||
        cudaMemcpyAsync(&status, h->check_status, sizeof(int), cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return SPMM_ERR_CUDA;
    }
    *host_status = status;
    return status == 0 ? SPMM_OK : SPMM_ERR_INVALID_CSR;
}

spmm_status_t spmm_measure_fp64_fma_rate(spmm_handle_t h, double* fma_per_second) {
    if (!h) return SPMM_ERR_INVALID_ARGUMENT;
    if (!fma_per_second) return SPMM_ERR_NULL_POINTER;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    // 32 warps per SM, 8 independent chains per thread: enough FMAs in flight
    // to cover the pipe's latency
    const int grid = 4 * h->num_sms;
    const int iters = 2048;
    spmm_status_t s = ensure_scratch(h, (size_t)grid * 256 * sizeof(double));
    if (s != SPMM_OK) return s;
    double* sink = static_cast<double*>(h->scratch);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        cudaGetLastError();
        if (e0) cudaEventDestroy(e0);
        return SPMM_ERR_CUDA;
    }
    cudaStream_t st = nullptr;
    int64_t fmas = 0;
    double best = 0.0;
    bool ok = launch_fp64_fma_probe(grid, iters, sink, st, &fmas) == cudaSuccess;   // warm-up
    for (int rep = 0; ok && rep < 3; ++rep) {
        ok = cudaEventRecord(e0, st) == cudaSuccess &&
             launch_fp64_fma_probe(grid, iters, sink, st, &fmas) == cudaSuccess &&
             cudaEventRecord(e1, st) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess;
        float ms = 0.0f;
        if (ok) ok = cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess && ms > 0.0f;
        if (ok) best = std::max(best, (double)fmas / (ms * 1e-3));
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (!ok) {
        cudaGetLastError();
        return SPMM_ERR_CUDA;
    }
    *fma_per_second = best;
    return SPMM_OK;
}

spmm_status_t spmm_set_profiling(spmm_handle_t h, int enable) {
    if (!h) return SPMM_ERR_INVALID_ARGUMENT;
    if (enable && !h->ev[0]) {
        int cur = -1;
        if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
            cudaGetLastError();
            return SPMM_ERR_INVALID_ARGUMENT;
        }
        for (auto& e : h->ev) {
            if (cudaEventCreate(&e) != cudaSuccess) {
                cudaGetLastError();
                return SPMM_ERR_CUDA;
            }
        }
    }
    h->profiling = enable != 0;
    return SPMM_OK;
}

spmm_status_t spmm_get_profile(spmm_handle_t h, spmm_profile_t* out) {
    if (!h || !h->have_profile) return SPMM_ERR_INVALID_ARGUMENT;
    if (!out) return SPMM_ERR_NULL_POINTER;
    if (cudaEventSynchronize(h->ev[4]) != cudaSuccess) {
        cudaGetLastError();
        return SPMM_ERR_CUDA;
    }
    spmm_profile_t p = h->prof;
    float t[4] = {0, 0, 0, 0};
    for (int i = 0; i < 4; ++i)
        if (cudaEventElapsedTime(&t[i], h->ev[i], h->ev[i + 1]) != cudaSuccess) {
            cudaGetLastError();
            return SPMM_ERR_CUDA;
        }
    p.prepass_ms = t[0];
    p.rows_ms = t[1];
    p.long_ms = t[2];
    p.fixup_ms = t[3];
    cudaEventElapsedTime(&p.total_ms, h->ev[0], h->ev[4]);
    if (h->prof_hdr) {
        int hdr[HDR_WORDS];
        if (cudaMemcpy(hdr, h->prof_hdr, sizeof(hdr), cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            return SPMM_ERR_CUDA;
        }
        p.rows_short = hdr[HDR_COUNT_SHORT];
        p.rows_medium = hdr[HDR_COUNT_MEDIUM];
        p.rows_long = hdr[HDR_COUNT_LONG];
        p.long_nnz = hdr[HDR_LONG_NNZ];
    }
    *out = p;
    return SPMM_OK;
}

spmm_status_t spmm_plan_create(spmm_handle_t h, spmm_plan_t* out, const int32_t* row_ptr,
                               int64_t m, int64_t k, int64_t n, int elem_size, void* stream) {
    if (!out) return SPMM_ERR_NULL_POINTER;
    *out = nullptr;
    if (!h || m < 0 || k < 0 || n < 0 || (elem_size != 4 && elem_size != 8))
        return SPMM_ERR_INVALID_ARGUMENT;
    if (m > (int64_t)INT_MAX - BIN_TILE || k > (int64_t)INT_MAX || n > (int64_t)INT_MAX)
        return SPMM_ERR_INVALID_ARGUMENT;
    if (m > 0 && !row_ptr) return SPMM_ERR_NULL_POINTER;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    spmm_plan_s* pl = new (std::nothrow) spmm_plan_s();
    if (!pl) return SPMM_ERR_ALLOC;
    pl->h = h;
    pl->device = h->device;
    pl->m = m;
    pl->k = k;
    pl->n = n;
    pl->es = elem_size;
    pl->long_grid = long_grid_of(h);
    const ScratchLayout L = layout_for(m, n, elem_size, pl->long_grid);
    if (cudaMalloc(&pl->scratch, L.total) != cudaSuccess) {
        cudaGetLastError();
        delete pl;
        return SPMM_ERR_ALLOC;
    }
    char* base = static_cast<char*>(pl->scratch);
    BinScratch bs{};
    bs.hdr = pl->hdr = reinterpret_cast<int*>(base + L.hdr);
    bs.tile_counts = reinterpret_cast<int*>(base + L.tile_counts);
    bs.tile_offsets = reinterpret_cast<int*>(base + L.tile_offsets);
    bs.rowlist = pl->rowlist = reinterpret_cast<int*>(base + L.rowlist);
    bs.med_pre = pl->med_pre = reinterpret_cast<int*>(base + L.med_pre);
    bs.long_pre = pl->long_pre = reinterpret_cast<int*>(base + L.long_pre);
    bs.long_cnt = pl->long_cnt = reinterpret_cast<int*>(base + L.long_cnt);
    pl->partials = base + L.partials;
    bin_geometry(m, &bs.items, &bs.tiles);
    // bins for 16-byte-aligned operands (the usual case); products issued with
    // other alignments use the same bins, which are valid for any geometry
    const Plan P = make_plan_es(h, k, n, elem_size, true);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (m > 0 && n > 0 && k > 0) {
        if (launch_binning(row_ptr, (int)m, P.short_max, P.long_min, bs, st, SPMM_PDL) !=
                cudaSuccess ||
            cudaMemcpyAsync(pl->hdr_host, pl->hdr, sizeof(pl->hdr_host), cudaMemcpyDeviceToHost,
                            st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(pl->scratch);
            delete pl;
            return SPMM_ERR_CUDA;
        }
    }
    *out = pl;
    return SPMM_OK;
}

spmm_status_t spmm_plan_destroy(spmm_plan_t pl) {
    if (!pl) return SPMM_OK;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != pl->device) cudaSetDevice(pl->device);
    cudaDeviceSynchronize();
    cudaFree(pl->scratch);
    if (cur >= 0 && cur != pl->device) cudaSetDevice(cur);
    cudaGetLastError();
    delete pl;
    return SPMM_OK;
}

spmm_status_t spmm_plan_order_rows(spmm_plan_t pl, const int32_t* row_ptr,
                                   const int32_t* col_idx, void* stream) {
    try {
        return plan_order_rows(pl, row_ptr, col_idx, stream, false, nullptr);
    } catch (const std::bad_alloc&) {          // no C++ exception crosses the C ABI
        return SPMM_ERR_ALLOC;
    }
}

spmm_status_t spmm_plan_order_rows_auto(spmm_plan_t pl, const int32_t* row_ptr,
                                        const int32_t* col_idx, void* stream, int32_t* applied) {
    try {
        return plan_order_rows(pl, row_ptr, col_idx, stream, true, applied);
    } catch (const std::bad_alloc&) {
        if (applied) *applied = 0;
        return SPMM_ERR_ALLOC;
    }
}

spmm_status_t spmm_plan_csr_f32(spmm_plan_t plan, float alpha, const int32_t* row_ptr,
                                const int32_t* col_idx, const float* values, const float* B,
                                int64_t ldb, float beta, float* C, int64_t ldc, void* stream) {
    return spmm_plan_impl<float>(plan, alpha, row_ptr, col_idx, values, B, ldb, beta, C, ldc,
                                 stream);
}

spmm_status_t spmm_plan_csr_f64(spmm_plan_t plan, double alpha, const int32_t* row_ptr,
                                const int32_t* col_idx, const double* values, const double* B,
                                int64_t ldb, double beta, double* C, int64_t ldc, void* stream) {
    return spmm_plan_impl<double>(plan, alpha, row_ptr, col_idx, values, B, ldb, beta, C, ldc,
                                  stream);
}

spmm_status_t spmm_set_l2_persistence(spmm_handle_t h, int64_t bytes) {
    if (!h) return SPMM_ERR_INVALID_ARGUMENT;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return SPMM_ERR_INVALID_ARGUMENT;
    }
    if (bytes == 0) {
        if (h->persist_bytes > 0) {
            cudaError_t e1 = cudaCtxResetPersistingL2Cache();
            cudaError_t e2 = cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, h->persist_prev);
            h->persist_bytes = 0;
            if (e1 != cudaSuccess || e2 != cudaSuccess) {
                cudaGetLastError();
                return SPMM_ERR_CUDA;
            }
        }
        return SPMM_OK;
    }
    if (h->persist_max <= 0 || h->window_max <= 0) return SPMM_ERR_UNSUPPORTED_DEVICE;
    const int64_t want = bytes < 0 ? h->persist_max : std::min(bytes, h->persist_max);
    if (h->persist_bytes == 0 &&
        cudaDeviceGetLimit(&h->persist_prev, cudaLimitPersistingL2CacheSize) != cudaSuccess) {
        cudaGetLastError();
        return SPMM_ERR_CUDA;
    }
    if (cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, (size_t)want) != cudaSuccess) {
        cudaGetLastError();
        return SPMM_ERR_CUDA;
    }
    h->persist_bytes = want;
    return SPMM_OK;
}

spmm_status_t spmm_csr_squared_f32(spmm_handle_t h, float alpha, const int32_t* row_ptr,
                                   const int32_t* col_idx, const float* values, int64_t m,
                                   const float* B, int64_t ldb, int64_t n, float beta, float* C,
                                   int64_t ldc, void* stream) {
    return spmm_squared_impl<float>(h, alpha, row_ptr, col_idx, values, m, B, ldb, n, beta, C,
                                    ldc, stream);
}

spmm_status_t spmm_csr_squared_f64(spmm_handle_t h, double alpha, const int32_t* row_ptr,
                                   const int32_t* col_idx, const double* values, int64_t m,
                                   const double* B, int64_t ldb, int64_t n, double beta,
                                   double* C, int64_t ldc, void* stream) {
    return spmm_squared_impl<double>(h, alpha, row_ptr, col_idx, values, m, B, ldb, n, beta, C,
                                     ldc, stream);
}

spmm_status_t spmm_plan_csr_squared_f32(spmm_plan_t plan, float alpha, const int32_t* row_ptr,
                                        const int32_t* col_idx, const float* values,
                                        const float* B, int64_t ldb, float beta, float* C,
                                        int64_t ldc, void* stream) {
    return spmm_plan_squared_impl<float>(plan, alpha, row_ptr, col_idx, values, B, ldb, beta, C,
                                         ldc, stream);
}

spmm_status_t spmm_plan_csr_squared_f64(spmm_plan_t plan, double alpha, const int32_t* row_ptr,
                                        const int32_t* col_idx, const double* values,
                                        const double* B, int64_t ldb, double beta, double* C,
                                        int64_t ldc, void* stream) {
    return spmm_plan_squared_impl<double>(plan, alpha, row_ptr, col_idx, values, B, ldb, beta,
                                          C, ldc, stream);
}

spmm_status_t spmm_fw_argmin_f32(spmm_handle_t h, int64_t n, int64_t k,
                                 const int32_t* k2b_row_ptr, const int32_t* k2b_col_idx,
                                 const float* k2b_values, const int32_t* t1_row_ptr,
                                 const int32_t* t1_col_idx, const float* t1_values,
                                 const int32_t* t2_row_ptr, const int32_t* t2_col_idx,
                                 const float* t2_values, const int32_t* b_row_ptr,
                                 const int32_t* b_col_idx, const float* b_values, float* min_val,
                                 int32_t* min_idx, float* gap, void* stream) {
    return spmm_fw_impl<float>(h, n, k, k2b_row_ptr, k2b_col_idx, k2b_values, t1_row_ptr,
                               t1_col_idx, t1_values, t2_row_ptr, t2_col_idx, t2_values,
                               b_row_ptr, b_col_idx, b_values, min_val, min_idx, gap, stream);
}

spmm_status_t spmm_fw_argmin_f64(spmm_handle_t h, int64_t n, int64_t k,
                                 const int32_t* k2b_row_ptr, const int32_t* k2b_col_idx,
                                 const double* k2b_values, const int32_t* t1_row_ptr,
                                 const int32_t* t1_col_idx, const double* t1_values,
                                 const int32_t* t2_row_ptr, const int32_t* t2_col_idx,
                                 const double* t2_values, const int32_t* b_row_ptr,
                                 const int32_t* b_col_idx, const double* b_values,
                                 double* min_val, int32_t* min_idx, double* gap, void* stream) {
    return spmm_fw_impl<double>(h, n, k, k2b_row_ptr, k2b_col_idx, k2b_values, t1_row_ptr,
                                t1_col_idx, t1_values, t2_row_ptr, t2_col_idx, t2_values,
                                b_row_ptr, b_col_idx, b_values, min_val, min_idx, gap, stream);
}

spmm_status_t spmm_ilu0_f32(spmm_handle_t h, int64_t n, int64_t nnz, const int32_t* row_ptr,
                            const int32_t* col_idx, float* values, int32_t* depth,
                            int32_t* status, void* stream) {
    return spmm_ilu0_impl<float>(h, n, nnz, row_ptr, col_idx, values, depth, status, stream);
}

spmm_status_t spmm_ilu0_f64(spmm_handle_t h, int64_t n, int64_t nnz, const int32_t* row_ptr,
                            const int32_t* col_idx, double* values, int32_t* depth,
                            int32_t* status, void* stream) {
    return spmm_ilu0_impl<double>(h, n, nnz, row_ptr, col_idx, values, depth, status, stream);
}

const char* spmm_status_string(spmm_status_t s) {
    switch (s) {
        case SPMM_OK: return "SPMM_OK";
        case SPMM_ERR_INVALID_ARGUMENT: return "SPMM_ERR_INVALID_ARGUMENT: invalid argument";
        case SPMM_ERR_DIMENSION_MISMATCH:
            return "SPMM_ERR_DIMENSION_MISMATCH: leading dimension smaller than the column count";
        case SPMM_ERR_NULL_POINTER: return "SPMM_ERR_NULL_POINTER: required pointer is NULL";
        case SPMM_ERR_UNSUPPORTED_DEVICE:
            return "SPMM_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 (sm_103) GPU";
        case SPMM_ERR_ALLOC: return "SPMM_ERR_ALLOC: scratch allocation failed";
        case SPMM_ERR_CUDA: return "SPMM_ERR_CUDA: CUDA runtime or launch error";
        case SPMM_ERR_INVALID_CSR: return "SPMM_ERR_INVALID_CSR: malformed CSR structure";
        case SPMM_ERR_TOO_LARGE:
            return "SPMM_ERR_TOO_LARGE: m or n beyond the static scratch of spmm_csr_f32_noalloc";
    }
    return "unknown spmm status";
}

}  // extern "C"
