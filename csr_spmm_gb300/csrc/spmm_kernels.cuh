// Per-bin CSR SpMM kernels, templated on
//   T  element type (float / double)
//   W  elements per B/C vector access (W * sizeof(T) = 16 bytes, or 1 element)
//   G  lanes per row group: a group of G lanes covers G * R * W columns of C,
//      one vector of W columns per lane and slot
//   R  vector slots per lane (wide panels: G = 32 and R > 1)
//
// The product for one output row i is acc[c] = sum_p values[p] * B[col_idx[p], c]
// over the row's entries p (oxicuda-sparse, ops/spmm.rs: module doc "Strategy"
// and the `spmm` kernel's nnz loop), followed by the alpha/beta epilogue.  The
// page's kernel gives one thread a row and a 4-column tile and re-reads the row
// once per column; here a lane group shares each (col_idx, value) pair by warp
// shuffle and every lane gathers a 16-byte vector of the B row, so each B row
// segment is fetched with full-sector, coalesced requests.
//
// Entry distribution: in each step a group takes CH = max(G, U) consecutive
// entries; lane g of the group loads entries g, g + G, ... of the step
// (coalesced), then the group walks them in batches of U, broadcasting
// (col, value) from the owning lane and issuing U * R independent B gathers
// before the FMAs, so that every lane keeps U * R loads in flight.
#pragma once

#include "spmm_device.cuh"

namespace spmm {

template <typename T, int W, int G, int R>
struct Cfg {
    static_assert(G >= 1 && G <= 32 && (G & (G - 1)) == 0, "G must be a power of two <= 32");
    static constexpr int SLOTS = G * R;                       // vectors per column pass
    static constexpr int BYTES_PER_ENTRY = R * W * (int)sizeof(T);
    static constexpr int U0 = 128 / BYTES_PER_ENTRY;          // ~128 B of loads in flight/lane
    static constexpr int U = U0 < 1 ? 1 : (U0 > 8 ? 8 : U0);  // entries per batch
    static constexpr int CH = G > U ? G : U;                  // entries per group per step
    static constexpr int Q = CH / G;                          // (col, value) loads per lane per step
    static constexpr int RPW = 32 / G;                        // groups (rows) per warp
};

// Accumulate entries [e0, e0 + len) of A into acc, for the column pass whose
// first vector is vbase, in a panel of pw columns starting at c0.
//   MEDIUM == false: each group walks its own row (e0, len per group); the
//                    step loop runs to the longest row in the warp.
//   MEDIUM == true : the whole warp shares one entry range; group gi takes
//                    entries [s + gi*CH, s + gi*CH + CH) of each warp step of
//                    RPW*CH entries.  The caller combines the groups.
template <typename T, int W, int G, int R, bool MEDIUM>
__device__ __forceinline__ void accumulate(T (&acc)[R][W], const int* __restrict__ col_idx,
                                           const T* __restrict__ values,
                                           const T* __restrict__ Bp, int64_t ldb, int e0,
                                           int len, int vbase, int pw, uint64_t pol_b,
                                           uint64_t pol_s) {
    using C = Cfg<T, W, G, R>;
    const int lane = threadIdx.x & 31;
    const int g = lane & (G - 1);
    const int gi = lane / G;
    const int step = MEDIUM ? C::RPW * C::CH : C::CH;
    const int goff = MEDIUM ? gi * C::CH : 0;
    const int span = MEDIUM ? len : __reduce_max_sync(FULL, len);   // warp-uniform

    for (int s = 0; s < span; s += step) {
        // load this step's (col, value) pairs: lane g holds entries g + G*q
        int colr[C::Q];
        T valr[C::Q];
#pragma unroll
        for (int q = 0; q < C::Q; ++q) {
            const int j = s + goff + g + G * q;
            colr[q] = 0;
            valr[q] = T(0);
            if (j < len) {
                colr[q] = ld_stream(col_idx + e0 + j, pol_s);
                valr[q] = ld_stream(values + e0 + j, pol_s);
            }
        }
        const int cnt = min(C::CH, len - s - goff);   // valid entries for this group (may be <= 0)
        const int cmax = min(C::CH, span - s);          // warp-uniform bound
#pragma unroll
        for (int j0 = 0; j0 < C::CH; j0 += C::U) {
            if (j0 >= cmax) break;                      // uniform
            T bv[C::U][R][W];
            T av[C::U];
#pragma unroll
            for (int u = 0; u < C::U; ++u) {
                const int j = j0 + u;                   // compile-time after unrolling
                const int q = (j / G) % C::Q;
                const int src = j % G;
                const int cj = __shfl_sync(FULL, colr[q], src, G);
                const T aj = __shfl_sync(FULL, valr[q], src, G);
                const bool ok = (j < C::CH) && (j < cnt);
                av[u] = ok ? aj : T(0);
                const T* brow = Bp + (int64_t)cj * ldb;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int col = (vbase + g + G * r) * W;
                    if (ok && col < pw) {
                        if (col + W <= pw) BLoad<T, W>::run(brow + col, bv[u][r], pol_b);
                        else load_b_partial<T, W>(brow + col, pw - col, bv[u][r], pol_b);
                    } else {
#pragma unroll
                        for (int e = 0; e < W; ++e) bv[u][r][e] = T(0);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < C::U; ++u)
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int e = 0; e < W; ++e) acc[r][e] = fma(av[u], bv[u][r][e], acc[r][e]);
        }
    }
}

// Sum the warp's groups (lanes g, g+G, g+2G, ...) with a fixed xor tree.
template <typename T, int W, int G, int R>
__device__ __forceinline__ void combine_groups(T (&acc)[R][W]) {
#pragma unroll
    for (int off = G; off < 32; off <<= 1)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < W; ++e) acc[r][e] += __shfl_xor_sync(FULL, acc[r][e], off);
}

template <typename T, int W, int G, int R>
__device__ __forceinline__ void write_row(T* __restrict__ Crow, const T (&acc)[R][W], int vbase,
                                          int pw, T alpha, T beta, bool read_c) {
    const int g = (threadIdx.x & 31) & (G - 1);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int col = (vbase + g + G * r) * W;
        if (col < pw) store_c<T, W>(Crow + col, min(W, pw - col), acc[r], alpha, beta, read_c);
    }
}

// ---------------------------------------------------------------------------
// Short and medium rows.  One persistent launch walks warp items, panel-major:
// per panel, first the short items (RPW rows each, one per lane group), then
// the medium rows (one warp each, groups split the entries).
// ---------------------------------------------------------------------------
template <typename T, int W, int G, int R>
__global__ void __launch_bounds__(ROWS_THREADS)
rows_kernel(SpmmParams<T> p) {
    using C = Cfg<T, W, G, R>;
    const int lane = threadIdx.x & 31;
    const int gi = lane / G;
    const uint64_t pol_b = policy_evict_last();
    const uint64_t pol_s = policy_evict_first();
    const int n_short = p.hdr[HDR_COUNT_SHORT];
    const int n_med = p.hdr[HDR_COUNT_MEDIUM];
    const int64_t items_short = (n_short + C::RPW - 1) / C::RPW;
    const int64_t items_panel = items_short + n_med;
    const int64_t total = items_panel * p.npanels;
    const int64_t nwarps = (int64_t)gridDim.x * (ROWS_THREADS / 32);
    const bool read_c = p.beta != T(0);

    for (int64_t it = (int64_t)blockIdx.x * (ROWS_THREADS / 32) + (threadIdx.x >> 5); it < total;
         it += nwarps) {
        const int panel = (int)(it / items_panel);
        const int64_t item = it - (int64_t)panel * items_panel;
        const int c0 = panel * p.panel_cols;
        const int pw = min(p.panel_cols, p.n - c0);
        const int nvec = (pw + W - 1) / W;
        const T* Bp = p.B + c0;
        if (item < items_short) {
            const int64_t idx = item * C::RPW + gi;
            const int row = idx < n_short ? p.rowlist[idx] : -1;
            int e0 = 0, len = 0;
            if (row >= 0) {
                e0 = p.row_ptr[row];
                len = p.row_ptr[row + 1] - e0;
            }
            for (int vbase = 0; vbase < nvec; vbase += C::SLOTS) {
                T acc[R][W];
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int e = 0; e < W; ++e) acc[r][e] = T(0);
                accumulate<T, W, G, R, false>(acc, p.col_idx, p.values, Bp, p.ldb, e0, len, vbase,
                                              pw, pol_b, pol_s);
                if (row >= 0)
                    write_row<T, W, G, R>(p.C + (int64_t)row * p.ldc + c0, acc, vbase, pw,
                                          p.alpha, p.beta, read_c);
            }
        } else {
            const int row = p.rowlist[n_short + (item - items_short)];
            const int e0 = p.row_ptr[row];
            const int len = p.row_ptr[row + 1] - e0;
            for (int vbase = 0; vbase < nvec; vbase += C::SLOTS) {
                T acc[R][W];
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int e = 0; e < W; ++e) acc[r][e] = T(0);
                accumulate<T, W, G, R, true>(acc, p.col_idx, p.values, Bp, p.ldb, e0, len, vbase,
                                             pw, pol_b, pol_s);
                combine_groups<T, W, G, R>(acc);
                if (gi == 0)
                    write_row<T, W, G, R>(p.C + (int64_t)row * p.ldc + c0, acc, vbase, pw,
                                          p.alpha, p.beta, read_c);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Long rows: deterministic CTA split.
// The long rows, concatenated in ascending row order, hold `total` entries.
// CTA c takes entries [c*seg, min((c+1)*seg, total)) with
// seg = max(ceil(total / long_grid), LONG_MIN_SEGMENT), a function of the data
// only.  For each long row overlapping its range, the CTA's warps split the
// overlap evenly, each warp's groups split it further, and the warp sums are
// added in warp order through shared memory.  A row lying wholly inside the
// range is finished here (epilogue to C).  Otherwise the CTA stores a partial
// sum: slot 0 for the row containing the range's first entry, slot 1 for the
// row containing its last; the fixup kernel adds the partials of each split
// row in CTA order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int long_segment(int total, int long_grid) {
    const int s = (int)(((int64_t)total + long_grid - 1) / long_grid);
    return s > LONG_MIN_SEGMENT ? s : LONG_MIN_SEGMENT;
}

template <typename T, int W, int G, int R>
__global__ void __launch_bounds__(LONG_THREADS)
long_kernel(SpmmParams<T> p) {
    using C = Cfg<T, W, G, R>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* red = reinterpret_cast<T*>(smem_raw);      // [LONG_WARPS][SLOTS * W]
    const int nl = p.hdr[HDR_COUNT_LONG];
    const int total = p.hdr[HDR_LONG_NNZ];
    if (nl == 0 || total == 0) return;
    const int seg = long_segment(total, p.long_grid);
    const int s0 = (int)min((int64_t)blockIdx.x * seg, (int64_t)total);
    if (s0 >= total) return;                      // uniform per CTA
    const int s1 = (int)min((int64_t)s0 + seg, (int64_t)total);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane & (G - 1), gi = lane / G;
    const uint64_t pol_b = policy_evict_last();
    const uint64_t pol_s = policy_evict_first();
    const bool read_c = p.beta != T(0);
    const int* lrows = p.rowlist + p.hdr[HDR_COUNT_SHORT] + p.hdr[HDR_COUNT_MEDIUM];

    // r0: the long row containing entry s0 (largest r with long_pre[r] <= s0)
    int lo = 0, hi = nl - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.long_pre[mid] <= s0) lo = mid; else hi = mid - 1;
    }
    const int r0 = lo;

    for (int panel = 0; panel < p.npanels; ++panel) {
        const int c0 = panel * p.panel_cols;
        const int pw = min(p.panel_cols, p.n - c0);
        const int nvec = (pw + W - 1) / W;
        const T* Bp = p.B + c0;
        for (int r = r0; r < nl; ++r) {
            const int pre_r = p.long_pre[r];
            if (pre_r >= s1) break;
            const int pre_r1 = p.long_pre[r + 1];
            const int a = max(s0, pre_r), b = min(s1, pre_r1);
            const int row = lrows[r];
            const int off = p.row_ptr[row] - pre_r;        // concatenated -> A entry index
            const int len = b - a;
            const int wl = a + off + (int)((int64_t)len * warp / LONG_WARPS);
            const int wh = a + off + (int)((int64_t)len * (warp + 1) / LONG_WARPS);
            const bool whole = pre_r >= s0 && pre_r1 <= s1;
            const int slot = (r == r0) ? 0 : 1;
            for (int vbase = 0; vbase < nvec; vbase += C::SLOTS) {
                T acc[R][W];
#pragma unroll
                for (int q = 0; q < R; ++q)
#pragma unroll
                    for (int e = 0; e < W; ++e) acc[q][e] = T(0);
                accumulate<T, W, G, R, true>(acc, p.col_idx, p.values, Bp, p.ldb, wl, wh - wl,
                                             vbase, pw, pol_b, pol_s);
                combine_groups<T, W, G, R>(acc);
                if (gi == 0) {
#pragma unroll
                    for (int q = 0; q < R; ++q)
#pragma unroll
                        for (int e = 0; e < W; ++e)
                            red[warp * (C::SLOTS * W) + (g + G * q) * W + e] = acc[q][e];
                }
                __syncthreads();
                if (warp == 0 && gi == 0) {
                    T sum[R][W];
#pragma unroll
                    for (int q = 0; q < R; ++q)
#pragma unroll
                        for (int e = 0; e < W; ++e) {
                            T s = T(0);
                            for (int w = 0; w < LONG_WARPS; ++w)
                                s += red[w * (C::SLOTS * W) + (g + G * q) * W + e];
                            sum[q][e] = s;
                        }
                    if (whole) {
                        write_row<T, W, G, R>(p.C + (int64_t)row * p.ldc + c0, sum, vbase, pw,
                                              p.alpha, p.beta, read_c);
                    } else {
                        T* dst = p.partials + ((int64_t)blockIdx.x * 2 + slot) * p.n + c0;
#pragma unroll
                        for (int q = 0; q < R; ++q) {
                            const int col = (vbase + g + G * q) * W;
#pragma unroll
                            for (int e = 0; e < W; ++e)
                                if (col + e < pw) dst[col + e] = sum[q][e];
                        }
                    }
                }
                __syncthreads();
            }
        }
    }
}

// Adds the partial sums of every long row that spans more than one CTA, in
// CTA order, and applies the epilogue.  One CTA per row (grid-stride).
template <typename T>
__global__ void __launch_bounds__(256)
fixup_kernel(SpmmParams<T> p) {
    const int nl = p.hdr[HDR_COUNT_LONG];
    const int total = p.hdr[HDR_LONG_NNZ];
    if (nl == 0 || total == 0) return;
    const int seg = long_segment(total, p.long_grid);
    const int* lrows = p.rowlist + p.hdr[HDR_COUNT_SHORT] + p.hdr[HDR_COUNT_MEDIUM];
    const bool read_c = p.beta != T(0);
    for (int r = blockIdx.x; r < nl; r += gridDim.x) {
        const int pre_r = p.long_pre[r], pre_r1 = p.long_pre[r + 1];
        const int cf = pre_r / seg, cl = (pre_r1 - 1) / seg;
        if (cf == cl) continue;                              // finished by its CTA
        const int slot_first = (pre_r == cf * seg) ? 0 : 1;
        const int row = lrows[r];
        T* Crow = p.C + (int64_t)row * p.ldc;
        for (int col = threadIdx.x; col < p.n; col += blockDim.x) {
            T s = p.partials[((int64_t)cf * 2 + slot_first) * p.n + col];
            for (int c = cf + 1; c <= cl; ++c) s += p.partials[((int64_t)c * 2) * p.n + col];
            const T o = read_c ? p.alpha * s + p.beta * Crow[col] : p.alpha * s;
            Crow[col] = o;
        }
    }
}

}  // namespace spmm
