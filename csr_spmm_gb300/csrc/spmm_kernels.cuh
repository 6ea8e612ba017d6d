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
// The kernels are bound by the latency of dependent memory round trips
// (row list -> row_ptr -> col_idx/values -> B), so each warp works through a
// contiguous range of rows with the stream software-pipelined: the row
// descriptors of 32 rows are loaded at once, and the (col_idx, value) pairs of
// the next step are in flight while the current step's B gathers are issued
// and consumed.
//
// Entry distribution: in each step a group takes CH = max(G, U) consecutive
// entries; lane g of the group holds entries g, g + G, ... of the step, and
// the group walks them in batches of U, broadcasting (col, value) from the
// owning lane and issuing U * R independent B gathers before the FMAs.
#pragma once

#include "spmm_device.cuh"

namespace spmm {

// binary32, 16-byte vectors, lane groups narrower than a warp
template <typename T, int W, int G>
constexpr bool narrow_f32() { return sizeof(T) == 4 && W * (int)sizeof(T) == 16 && G < 32; }

// ROWS: the short/medium-row kernel (narrow binary32 groups take the larger
// batch there; the long-row kernel keeps the general one).
template <typename T, int W, int G, int R, bool ROWS = false>
struct Cfg {
    static_assert(G >= 1 && G <= 32 && (G & (G - 1)) == 0, "G must be a power of two <= 32");
    static constexpr int SLOTS = G * R;                       // vectors per column pass
    static constexpr int BYTES_PER_ENTRY = R * W * (int)sizeof(T);
    static constexpr int BATCH_BYTES = sizeof(T) == 8 ? SPMM_BATCH_BYTES_F64
                                       : !ROWS                   ? SPMM_LONG_BATCH_BYTES
                                       : narrow_f32<T, W, G>()   ? SPMM_BATCH_BYTES_NARROW
                                                                 : SPMM_BATCH_BYTES;
    static constexpr int U0 = BATCH_BYTES / BYTES_PER_ENTRY;        // B bytes in flight/lane
    static constexpr int U = U0 < 1 ? 1 : (U0 > SPMM_BATCH_MAX ? SPMM_BATCH_MAX : U0);
    static constexpr int CH = G > U ? G : U;                  // entries per group per step
    static constexpr int Q = CH / G;                          // (col, value) loads per lane per step
    static constexpr int RPW = 32 / G;                        // groups per warp
    static_assert(CH % U == 0, "a step must hold whole batches");
};

template <typename T, int W, int R>
__device__ __forceinline__ void zero_acc(T (&acc)[R][W]) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < W; ++e) acc[r][e] = T(0);
}

// Lane g of a group loads entries first + g + G*q (q < Q) that lie below `limit`.
template <typename T, int G, int Q>
__device__ __forceinline__ void load_entries(int (&col)[Q], T (&val)[Q],
                                             const int* __restrict__ col_idx,
                                             const T* __restrict__ values, int first, int limit,
                                             uint64_t pol_s) {
    const int g = (threadIdx.x & 31) & (G - 1);
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int j = first + g + G * q;
        col[q] = 0;
        val[q] = T(0);
        if (j < limit) {
            col[q] = ld_stream(col_idx + j, pol_s);
            val[q] = ld_stream(values + j, pol_s);
        }
    }
}

// This lane's B vectors in one column pass: where each of its R vectors
// starts (panel base + element offset) and how many of its W elements lie in
// the panel.  A lane whose vector starts past the panel's last column re-reads
// the panel's last vector instead: those addresses fall in the lines the other
// lanes of the row fetch anyway, so they add no traffic, and that lane's sums
// are never stored.  Every gather of a valid entry is then unpredicated.
template <typename T, int W, int R>
struct LaneVecs {
    const T* base[R];
    int cnt[R];
};

template <typename T, int W, int G, int R>
__device__ __forceinline__ LaneVecs<T, W, R> lane_vecs(const T* __restrict__ Bp, int vbase,
                                                       int pw) {
    const int g = (threadIdx.x & 31) & (G - 1);
    const int last = ((pw - 1) / W) * W;
    LaneVecs<T, W, R> lv;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int c = (vbase + g + G * r) * W;
        const int ce = c < pw ? c : last;
        lv.base[r] = Bp + ce;
        lv.cnt[r] = min(W, pw - ce);
    }
    return lv;
}

// WHOLE: every lane vector of the geometry is whole (n a multiple of W), so
// the partial-vector path is compiled out.
template <typename T, int W, bool WHOLE>
__device__ __forceinline__ void gather_b(const T* p, int cnt, T (&v)[W]) {
    if (WHOLE || W == 1 || cnt == W) BLoad<T, W>::run(p, v);
    else load_b_partial<T, W>(p, cnt, v);
}

// Broadcast of a step's (col_idx, value) pairs to every lane of the group.
// With warp shuffles a binary64 pair costs three shuffles (the index and the
// value's two halves), each one L1 data-pipe wavefront per group.  In the
// binary64 rows kernel (groups of 8 or more lanes) each step's pairs are
// instead staged in a per-group shared-memory slot, and every lane reads a
// pair with one 16-byte broadcast load.  Measured on GB300: Laplacian 0.216 ->
// 0.207 ms per call.  For binary32 the same staging (two pairs per 16-byte
// load) was slower (SEACells +5%, power-law +5%, wide-N +38%; more spills),
// so binary32 and the long-row kernel keep the shuffles.
template <typename T, int W, int G, int R, bool ROWS>
struct Bcast {
    static constexpr bool SMEM = ROWS && sizeof(T) == 8 && G >= 8;
    static constexpr int PAIR_BYTES = 16;             // {col_idx, pad, value}
    // per-group slot; the 16-byte pad staggers the groups' banks
    static constexpr int GROUP_BYTES = Cfg<T, W, G, R, ROWS>::CH * PAIR_BYTES + 16;
    static constexpr int WARP_BYTES = SMEM ? Cfg<T, W, G, R, ROWS>::RPW * GROUP_BYTES : 0;
};

// Store this lane's pairs of the step (entries g + G*q) in the group's slot.
template <int G, int Q>
__device__ __forceinline__ void stage_entries(unsigned char* slot, const int (&col)[Q],
                                              const double (&val)[Q]) {
    const int g = (threadIdx.x & 31) & (G - 1);
#pragma unroll
    for (int q = 0; q < Q; ++q)
        *reinterpret_cast<double2*>(slot + (g + G * q) * 16) =
            make_double2(__hiloint2double(0, col[q]), val[q]);
}

// Pair j of the step, for every lane of the group.
template <typename T, int W, int G, int R, bool ROWS>
__device__ __forceinline__ void fetch_pair(int& cj, T& av, int j,
                                           const int (&col)[Cfg<T, W, G, R, ROWS>::Q],
                                           const T (&val)[Cfg<T, W, G, R, ROWS>::Q],
                                           const unsigned char* slot) {
    if constexpr (Bcast<T, W, G, R, ROWS>::SMEM) {
        const double2 e = *reinterpret_cast<const double2*>(slot + j * 16);
        cj = __double2loint(e.x);
        av = e.y;
    } else {
        cj = __shfl_sync(FULL, col[j / G], j % G, G);   // j is compile-time after unrolling
        av = __shfl_sync(FULL, val[j / G], j % G, G);
    }
}

// The column of pair j alone, and its value alone.  In the binary32 kernels
// with lane groups narrower than a warp the value is broadcast when its FMAs
// run, not while the gathers are in flight, so it holds no register across
// the gather latency: fewer spills, power-law 0.874 -> 0.863 ms and wide-N
// 0.684 -> 0.678 ms per call on GB300, the same bits.  Full-warp groups keep
// the early broadcast (SEACells: 0.244 -> 0.287 ms with the late one).
template <typename T, int W, int G, int R, bool ROWS>
__device__ __forceinline__ int fetch_col(int j, const int (&col)[Cfg<T, W, G, R, ROWS>::Q],
                                         const unsigned char* slot) {
    if constexpr (Bcast<T, W, G, R, ROWS>::SMEM)
        return __double2loint(reinterpret_cast<const double2*>(slot + j * 16)->x);
    else
        return __shfl_sync(FULL, col[j / G], j % G, G);
}
template <typename T, int W, int G, int R, bool ROWS>
__device__ __forceinline__ T fetch_val(int j, const T (&val)[Cfg<T, W, G, R, ROWS>::Q],
                                       const unsigned char* slot) {
    if constexpr (Bcast<T, W, G, R, ROWS>::SMEM)
        return reinterpret_cast<const double2*>(slot + j * 16)->y;
    else
        return __shfl_sync(FULL, val[j / G], j % G, G);
}
#ifndef SPMM_LATE_VALUE
#define SPMM_LATE_VALUE 1
#endif
template <typename T, int W, int G>
constexpr bool late_value() { return SPMM_LATE_VALUE && narrow_f32<T, W, G>(); }

// One step: the group consumes its `cnt` (<= CH) entries held in (col, val),
// in batches of U.  cmax / cmin are warp-uniform bounds on every group's cnt:
// batches below cmin are whole for every group and gather without checks.
// Entries past a row's end were loaded with value 0 (load_entries).  `slot`
// is the group's shared-memory slot when Bcast::SMEM (every lane of the warp
// must call this together), unused otherwise.
template <typename T, int W, int G, int R, bool ROWS = false, bool WHOLE = false>
__device__ __forceinline__ void consume_step(T (&acc)[R][W],
                                             const int (&col)[Cfg<T, W, G, R, ROWS>::Q],
                                             const T (&val)[Cfg<T, W, G, R, ROWS>::Q], int cnt,
                                             int cmax, int cmin, int ldb,
                                             const LaneVecs<T, W, R>& lv,
                                             unsigned char* slot = nullptr) {
    using C = Cfg<T, W, G, R, ROWS>;
    if constexpr (Bcast<T, W, G, R, ROWS>::SMEM) {
        __syncwarp();                                   // the previous step's reads are done
        stage_entries<G, C::Q>(slot, col, val);
        __syncwarp();
    }
#pragma unroll
    for (int j0 = 0; j0 < C::CH; j0 += C::U) {
        if (j0 >= cmax) break;                          // warp-uniform
        T bv[C::U][R][W];
        T av[C::U];
        if (j0 + C::U <= cmin) {                        // warp-uniform: whole batch
#pragma unroll
            for (int u = 0; u < C::U; ++u) {
                int cj;
                if constexpr (late_value<T, W, G>())
                    cj = fetch_col<T, W, G, R, ROWS>(j0 + u, col, slot);
                else
                    fetch_pair<T, W, G, R, ROWS>(cj, av[u], j0 + u, col, val, slot);
                const int64_t roff = (int64_t)cj * ldb;
#pragma unroll
                for (int r = 0; r < R; ++r)
                    gather_b<T, W, WHOLE>(lv.base[r] + roff, lv.cnt[r], bv[u][r]);
            }
        } else {
#pragma unroll
            for (int u = 0; u < C::U; ++u) {
                const int j = j0 + u;
                int cj;
                if constexpr (late_value<T, W, G>())
                    cj = fetch_col<T, W, G, R, ROWS>(j, col, slot);
                else
                    fetch_pair<T, W, G, R, ROWS>(cj, av[u], j, col, val, slot);
                const int64_t roff = (int64_t)cj * ldb;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (j < cnt) {
                        gather_b<T, W, WHOLE>(lv.base[r] + roff, lv.cnt[r], bv[u][r]);
                    } else {
#pragma unroll
                        for (int e = 0; e < W; ++e) bv[u][r][e] = T(0);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < C::U; ++u) {
            if constexpr (late_value<T, W, G>())
                av[u] = fetch_val<T, W, G, R, ROWS>(j0 + u, val, slot);
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
                                          int pw, T alpha, T beta, bool read_c, bool keep = false) {
    const int g = (threadIdx.x & 31) & (G - 1);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int col = (vbase + g + G * r) * W;
        if (col < pw)
            store_c<T, W>(Crow + col, min(W, pw - col), acc[r], alpha, beta, read_c, keep);
    }
}

// The C row a lane group will update (beta != 0), loaded when the group
// starts the row so that the load overlaps the row's gathers.
template <typename T, int W, int G, int R>
__device__ __forceinline__ void load_c_row(T (&c0)[R][W], const T* __restrict__ Crow, int vbase,
                                           int pw) {
    const int g = (threadIdx.x & 31) & (G - 1);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int col = (vbase + g + G * r) * W;
#pragma unroll
        for (int e = 0; e < W; ++e) c0[r][e] = T(0);
        if (col < pw) load_c<T, W>(Crow + col, min(W, pw - col), c0[r]);
    }
}

template <typename T, int W, int G, int R, int BS>
__device__ __forceinline__ void write_row_c0(T* __restrict__ Crow, const T (&acc)[R][W],
                                             const T (&c0)[R][W], int vbase, int pw, T alpha,
                                             T beta) {
    const int g = (threadIdx.x & 31) & (G - 1);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int col = (vbase + g + G * r) * W;
        if (col < pw)
            store_c_pre<T, W, BS>(Crow + col, min(W, pw - col), acc[r], c0[r], alpha, beta);
    }
}

// ---------------------------------------------------------------------------
// A warp works through rows list[first + i * stride], i < count, of one bin,
// for the panel of pw columns starting at c0col.
//   MEDIUM == false (short rows): group gi takes rows gi, gi + RPW, ... of
//     every 32-row block; each group walks its own row CH entries per step.
//   MEDIUM == true (medium rows): the whole warp takes one row at a time;
//     group gi takes entries [s + gi*CH, s + gi*CH + CH) of each warp step of
//     RPW*CH entries, and the groups are combined at the end of the row.
// ---------------------------------------------------------------------------
// ext (the one-launch path): each row's (first entry, length), indexed by row,
// already in shared memory, in place of two row_ptr reads per row.
template <typename T, int W, int G, int R, bool MEDIUM, bool READ_C, bool WHOLE, int BS>
__device__ __forceinline__ void process_rows(const SpmmParams<T>& p, const int* __restrict__ list,
                                             int first, int count, int stride, int c0col, int pw,
                                             uint64_t pol_s, unsigned char* wslot,
                                             const int2* ext = nullptr) {
    using C = Cfg<T, W, G, R, true>;
    constexpr int Q = C::Q;
    const int lane = threadIdx.x & 31;
    const int gi = lane / G;
    constexpr int TSTEP = MEDIUM ? 1 : C::RPW;              // row-slot advance per row
    constexpr int ESTEP = MEDIUM ? C::RPW * C::CH : C::CH;  // entry advance per step
    const int goff = MEDIUM ? gi * C::CH : 0;
    unsigned char* slot = wslot + gi * Bcast<T, W, G, R, true>::GROUP_BYTES;
    const int nvec = (pw + W - 1) / W;
    const T* Bp = p.B + c0col;
    const int ldb = (int)p.ldb;                            // <= INT_MAX (host check)

    for (int sub = 0; sub < count; sub += 32) {
        const int nrows = min(32, count - sub);
        int my_row = -1, my_e0 = 0, my_len = 0;
        if (lane < nrows) {
            my_row = list[first + (int64_t)(sub + lane) * stride];
            if (ext) {
                const int2 x = ext[my_row];
                my_e0 = x.x;
                my_len = x.y;
            } else {
                my_e0 = p.row_ptr[my_row];
                my_len = p.row_ptr[my_row + 1] - my_e0;
            }
        }
        for (int vbase = 0; vbase < nvec; vbase += C::SLOTS) {
            const LaneVecs<T, W, R> lv = lane_vecs<T, W, G, R>(Bp, vbase, pw);
            int t = MEDIUM ? 0 : gi;
            int row = __shfl_sync(FULL, my_row, t & 31);
            int e0 = __shfl_sync(FULL, my_e0, t & 31);
            const int len0 = __shfl_sync(FULL, my_len, t & 31);
            int len = t < nrows ? len0 : 0;
            int s = 0;
            T acc[R][W];
            zero_acc<T, W, R>(acc);
            T c0[R][W];
            zero_acc<T, W, R>(c0);
            const bool loads_c = READ_C && (!MEDIUM || gi == 0);
            if (loads_c && t < nrows)
                load_c_row<T, W, G, R>(c0, p.C + (int64_t)row * p.ldc + c0col, vbase, pw);
            int colc[Q];
            T valc[Q];
            load_entries<T, G, Q>(colc, valc, p.col_idx, p.values, e0 + goff, e0 + len, pol_s);

            while (__any_sync(FULL, t < nrows)) {
                const bool active = t < nrows;
                // next position of this group, and its entries (prefetch)
                int t2 = t, s2 = s + ESTEP;
                if (s2 >= len) {
                    t2 = t + TSTEP;
                    s2 = 0;
                }
                const int row2 = __shfl_sync(FULL, my_row, t2 & 31);
                const int e02 = __shfl_sync(FULL, my_e0, t2 & 31);
                const int lraw = __shfl_sync(FULL, my_len, t2 & 31);
                const int len2 = t2 < nrows ? lraw : 0;
                int coln[Q];
                T valn[Q];
                load_entries<T, G, Q>(coln, valn, p.col_idx, p.values, e02 + s2 + goff,
                                      e02 + len2, pol_s);

                // consume the current step
                const int cnt = active ? min(C::CH, len - s - goff) : 0;
                int cmax, cmin;
                if constexpr (MEDIUM) {                    // groups staggered by CH entries
                    cmax = min(C::CH, len - s);
                    cmin = max(0, min(C::CH, len - s - (C::RPW - 1) * C::CH));
                } else if constexpr (G == 32) {            // one group: cnt is warp-uniform
                    cmax = cmin = max(cnt, 0);
                } else {
                    cmax = (int)__reduce_max_sync(FULL, (unsigned)max(cnt, 0));
                    cmin = (int)__reduce_min_sync(FULL, (unsigned)max(cnt, 0));
                }
                consume_step<T, W, G, R, true, WHOLE>(acc, colc, valc, cnt, cmax, cmin, ldb, lv,
                                                      slot);

                if (s + ESTEP >= len) {                     // row finished (uniform if MEDIUM)
                    if (MEDIUM) combine_groups<T, W, G, R>(acc);
                    if (active && (!MEDIUM || gi == 0)) {
                        T* Crow = p.C + (int64_t)row * p.ldc + c0col;
                        if constexpr (READ_C)
                            write_row_c0<T, W, G, R, BS>(Crow, acc, c0, vbase, pw, p.alpha,
                                                         p.beta);
                        else
                            write_row<T, W, G, R>(Crow, acc, vbase, pw, p.alpha, p.beta, false,
                                                  p.keep_c);
                    }
                    zero_acc<T, W, R>(acc);
                    if (loads_c && t2 < nrows)
                        load_c_row<T, W, G, R>(c0, p.C + (int64_t)row2 * p.ldc + c0col, vbase, pw);
                }
                t = t2;
                s = s2;
                row = row2;
                e0 = e02;
                len = len2;
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    colc[q] = coln[q];
                    valc[q] = valn[q];
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Short and medium rows.  Persistent launch: for each panel (in order), warp w
// takes the w-th of nwarps equal contiguous ranges of the short list, then of
// the medium list.
// ---------------------------------------------------------------------------
// First medium row whose entries start at or after `target` (lower bound in
// the medium-length prefix).
__device__ __forceinline__ int medium_lower_bound(const int* __restrict__ med_pre, int n_med,
                                                  int64_t target) {
    int lo = 0, hi = n_med;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)med_pre[mid] < target) lo = mid + 1; else hi = mid;
    }
    return lo;
}

#ifndef SPMM_SHORT_INTERLEAVE
#define SPMM_SHORT_INTERLEAVE 1
#endif

template <typename T, int W, int G>
struct RowsOccupancy {
    static constexpr int THREADS = sizeof(T) == 8 ? SPMM_ROWS_THREADS_F64
                                   : narrow_f32<T, W, G>() ? SPMM_ROWS_THREADS_NARROW
                                                           : SPMM_ROWS_THREADS;
    static constexpr int MIN_BLOCKS = sizeof(T) == 8 ? SPMM_ROWS_MIN_BLOCKS_F64
                                      : narrow_f32<T, W, G>() ? SPMM_ROWS_MIN_BLOCKS_NARROW
                                                              : SPMM_ROWS_MIN_BLOCKS;
    static_assert(THREADS % 32 == 0 && THREADS <= 1024, "rows kernel block size");
};

// READ_C: beta != 0 (C is read, and prefetched at each row start).
// WHOLE: n is a multiple of W (no partial vectors; see gather_b).
// BS: 0 for any beta; +1 / -1 for a launch with beta == +1 / -1 (see epi).
template <typename T, int W, int G, int R, bool READ_C, bool WHOLE, int BS = 0>
__global__ void __launch_bounds__(RowsOccupancy<T, W, G>::THREADS, RowsOccupancy<T, W, G>::MIN_BLOCKS)
rows_kernel(SpmmParams<T> p) {
    constexpr int WPB = RowsOccupancy<T, W, G>::THREADS / 32;    // warps per block
    // per-warp slots for the (col_idx, value) broadcast (Bcast)
    constexpr int SLOT_BYTES = Bcast<T, W, G, R, true>::WARP_BYTES;
    __shared__ __align__(16) unsigned char s_slots[SLOT_BYTES > 0 ? WPB * SLOT_BYTES : 16];
    unsigned char* wslot = s_slots + (threadIdx.x >> 5) * SLOT_BYTES;
    wait_for_predecessor();
    allow_successor();
    const uint64_t pol_s = policy_evict_first();
    const int n_short = p.hdr[HDR_COUNT_SHORT];
    const int n_med = p.hdr[HDR_COUNT_MEDIUM];
    const int64_t med_nnz = p.hdr[HDR_MED_NNZ];
    const int64_t nwarps = (int64_t)gridDim.x * WPB;
    const int64_t w = (int64_t)blockIdx.x * WPB + (threadIdx.x >> 5);
    // short rows: equal counts per warp; medium rows: equal entries per warp
    // short rows: each CTA takes an equal contiguous range of the short list and
    // its warps interleave over it (warp j: rows j, j + WPB, ...), so rows that
    // sit next to each other in the list run at the same time on the same SM
    const int64_t nblk = gridDim.x;
    const int cs0 = (int)((int64_t)blockIdx.x * n_short / nblk);
    const int cs1 = (int)((int64_t)(blockIdx.x + 1) * n_short / nblk);
    const int wib = threadIdx.x >> 5;
    const int s_first = SPMM_SHORT_INTERLEAVE ? cs0 + wib : (int)(w * n_short / nwarps);
    const int s_count = SPMM_SHORT_INTERLEAVE
                            ? max(0, (cs1 - cs0 - wib + WPB - 1) / WPB)
                            : (int)((w + 1) * n_short / nwarps) - (int)(w * n_short / nwarps);
    const int s_stride = SPMM_SHORT_INTERLEAVE ? WPB : 1;
    int m0 = 0, m1 = 0;
    if (n_med > 0) {
        m0 = medium_lower_bound(p.med_pre, n_med, w * med_nnz / nwarps);
        m1 = medium_lower_bound(p.med_pre, n_med, (w + 1) * med_nnz / nwarps);
        if (w == nwarps - 1) m1 = n_med;
    }
    for (int panel = 0; panel < p.npanels; ++panel) {
        const int c0 = panel * p.panel_cols;
        const int pw = min(p.panel_cols, p.n - c0);
        if (s_count > 0)
            process_rows<T, W, G, R, false, READ_C, WHOLE, BS>(p, p.rowlist, s_first, s_count,
                                                               s_stride, c0, pw, pol_s, wslot);
        if (m1 > m0)
            process_rows<T, W, G, R, true, READ_C, WHOLE, BS>(p, p.rowlist + n_short, m0,
                                                              m1 - m0, 1, c0, pw, pol_s, wslot);
    }
}

// ---------------------------------------------------------------------------
// Small products (m <= SMALL_ROWS rows): the whole product in one launch.
// Every CTA bins all m rows itself in shared memory (their lengths are at
// most 8 KB of row_ptr, read from L2), so no pre-pass launch and no global
// bins are needed.  Short rows (<= short_max entries, the same threshold as
// the binned path) are then processed as in rows_kernel: CTA c takes an
// equal contiguous range of the short list and its warps interleave over it.
// Every longer row is processed by one warp, as a medium row of rows_kernel
// (the warp's groups split its entries and are combined at the row's end);
// the grid's warps take equal shares of those rows' entries.  Short and
// medium rows therefore give rows_kernel's results bit for bit; a row of
// long_min or more entries, which the binned path splits across CTAs, is
// summed in the medium-row order instead.  Rows keep their order in both
// lists (stable scans).
// ---------------------------------------------------------------------------
// Exclusive scan of v over the block (blockDim.x threads, a multiple of 32,
// at most 1024); returns this thread's prefix and sets *total.  s_warp holds
// 33 ints: the warps' prefixes, then the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* s_warp) {
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(FULL, incl, off);
        if (lane >= off) incl += y;
    }
    __syncthreads();                                   // s_warp free from any earlier scan
    if (lane == 31) s_warp[wib] = incl;
    __syncthreads();
    if (wib == 0) {
        int w = lane < nw ? s_warp[lane] : 0;
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(FULL, wi, off);
            if (lane >= off) wi += y;
        }
        if (lane < nw) s_warp[lane] = wi - w;          // exclusive prefix of warp totals
        if (lane == 31) s_warp[32] = wi;               // block total
    }
    __syncthreads();
    *total = s_warp[32];
    return s_warp[wib] + incl - v;
}

template <typename T, int W, int G, int R, bool READ_C, bool WHOLE, int BS = 0>
__global__ void __launch_bounds__(RowsOccupancy<T, W, G>::THREADS, 1)
small_kernel(SpmmParams<T> p, int short_max) {
    constexpr int THREADS = RowsOccupancy<T, W, G>::THREADS;
    constexpr int WPB = THREADS / 32;
    static_assert(WPB <= 32, "one scan word per warp");
    constexpr int SLOT_BYTES = Bcast<T, W, G, R, true>::WARP_BYTES;
    __shared__ __align__(16) unsigned char s_slots[SLOT_BYTES > 0 ? WPB * SLOT_BYTES : 16];
    // short rows ascending from the front; longer rows from the back, the
    // j-th longer row (ascending) at SMALL_ROWS - 1 - j
    __shared__ int s_list[SMALL_ROWS];
    __shared__ int s_pre[SMALL_ROWS + 1];   // exclusive prefix of the longer rows' lengths
    __shared__ int2 s_ext[SMALL_ROWS];      // every row's first entry and length
    __shared__ int s_warp[33];
    unsigned char* wslot = s_slots + (threadIdx.x >> 5) * SLOT_BYTES;
    const int m = p.m;

    // every row's extents, and whether all rows are short
    bool all_short = true;
    for (int r = (int)threadIdx.x; r < m; r += THREADS) {
        const int e0 = p.row_ptr[r];
        const int len = p.row_ptr[r + 1] - e0;
        s_ext[r] = make_int2(e0, len);
        all_short &= len <= short_max;
    }
    all_short = __syncthreads_and(all_short);
    int n_short = 0, n_other = 0, other_nnz = 0;     // block-uniform
    if (all_short) {
        for (int r = (int)threadIdx.x; r < m; r += THREADS) s_list[r] = r;
        n_short = m;
    } else {
        // stable ranks, chunk by chunk, by block scans
        for (int c0 = 0; c0 < m; c0 += THREADS) {
            const int r = c0 + (int)threadIdx.x;
            const int len = r < m ? s_ext[r].y : 0;
            const bool is_short = r < m && len <= short_max;
            const bool is_other = r < m && !is_short;
            int tot_s, tot_o, tot_e;
            const int rank_s = block_exclusive_scan(is_short ? 1 : 0, &tot_s, s_warp);
            const int rank_o = block_exclusive_scan(is_other ? 1 : 0, &tot_o, s_warp);
            const int pre_e = block_exclusive_scan(is_other ? len : 0, &tot_e, s_warp);
            if (is_short) s_list[n_short + rank_s] = r;
            if (is_other) {
                s_list[SMALL_ROWS - 1 - (n_other + rank_o)] = r;
                s_pre[n_other + rank_o] = other_nnz + pre_e;
            }
            n_short += tot_s;
            n_other += tot_o;
            other_nnz += tot_e;
        }
        if (threadIdx.x == 0) s_pre[n_other] = other_nnz;
    }
    __syncthreads();

    const uint64_t pol_s = policy_evict_first();
    const int wib = threadIdx.x >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * WPB;
    const int64_t w = (int64_t)blockIdx.x * WPB + wib;
    // short rows: an equal contiguous range per CTA, the CTA's warps interleaved
    const int cs0 = (int)((int64_t)blockIdx.x * n_short / gridDim.x);
    const int cs1 = (int)((int64_t)(blockIdx.x + 1) * n_short / gridDim.x);
    const int s_count = max(0, (cs1 - cs0 - wib + WPB - 1) / WPB);
    // longer rows: equal shares of their entries per warp of the grid
    int o0 = 0, o1 = 0;
    if (n_other > 0) {
        o0 = medium_lower_bound(s_pre, n_other, w * other_nnz / nwarps);
        o1 = medium_lower_bound(s_pre, n_other, (w + 1) * other_nnz / nwarps);
        if (w == nwarps - 1) o1 = n_other;
    }
    for (int panel = 0; panel < p.npanels; ++panel) {
        const int c0 = panel * p.panel_cols;
        const int pw = min(p.panel_cols, p.n - c0);
        if (s_count > 0)
            process_rows<T, W, G, R, false, READ_C, WHOLE, BS>(p, s_list, cs0 + wib, s_count, WPB,
                                                               c0, pw, pol_s, wslot, s_ext);
        if (o1 > o0)      // longer row j at SMALL_ROWS - 1 - j: a descending walk of s_list
            process_rows<T, W, G, R, true, READ_C, WHOLE, BS>(p, s_list, SMALL_ROWS - 1 - o0,
                                                              o1 - o0, -1, c0, pw, pol_s, wslot,
                                                              s_ext);
    }
}

// ---------------------------------------------------------------------------
// Accumulate the entries [a, b) of one row, whole warp (groups interleaved as
// in the medium-row mode), with the next step's entries prefetched.  The
// caller combines the groups.
// ---------------------------------------------------------------------------
template <typename T, int W, int G, int R>
__device__ __forceinline__ void accumulate_range(T (&acc)[R][W], const SpmmParams<T>& p, int a,
                                                 int b, const T* __restrict__ Bp, int vbase,
                                                 int pw, uint64_t pol_s) {
    using C = Cfg<T, W, G, R>;
    constexpr int Q = C::Q;
    constexpr int ESTEP = C::RPW * C::CH;
    const int gi = (threadIdx.x & 31) / G;
    const int goff = gi * C::CH;
    const int ldb = (int)p.ldb;                            // <= INT_MAX (host check)
    const LaneVecs<T, W, R> lv = lane_vecs<T, W, G, R>(Bp, vbase, pw);
    int colc[Q];
    T valc[Q];
    load_entries<T, G, Q>(colc, valc, p.col_idx, p.values, a + goff, b, pol_s);
    for (int s = a; s < b; s += ESTEP) {
        int coln[Q];
        T valn[Q];
        load_entries<T, G, Q>(coln, valn, p.col_idx, p.values, s + ESTEP + goff, b, pol_s);
        const int cnt = min(C::CH, b - s - goff);
        const int cmax = min(C::CH, b - s);
        const int cmin = max(0, min(C::CH, b - s - (C::RPW - 1) * C::CH));
        consume_step<T, W, G, R>(acc, colc, valc, cnt, cmax, cmin, ldb, lv);
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            colc[q] = coln[q];
            valc[q] = valn[q];
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
// row containing its last; the last CTA to finish a split row adds its
// partials in CTA order (the fixup pass, in the same launch).
// ---------------------------------------------------------------------------
// Sum the partials of split long row r in CTA order (cf's slot, then slot 0
// of cf+1 .. cl) and apply the epilogue; every thread of the CTA takes
// columns threadIdx.x, threadIdx.x + blockDim.x, ...  Partials were written by
// other SMs, so they are read from L2 (ld.cg), never from a stale L1 line.
template <typename T>
__device__ __forceinline__ void finish_split_row(const SpmmParams<T>& p, const int* lrows, int r,
                                                 int seg, bool read_c) {
    const int pre_r = p.long_pre[r], pre_r1 = p.long_pre[r + 1];
    const int cf = pre_r / seg, cl = (pre_r1 - 1) / seg;
    const int slot_first = (pre_r == cf * seg) ? 0 : 1;
    T* Crow = p.C + (int64_t)lrows[r] * p.ldc;
    for (int col = threadIdx.x; col < p.n; col += blockDim.x) {
        T s = __ldcg(p.partials + ((int64_t)cf * 2 + slot_first) * p.n + col);
        for (int c = cf + 1; c <= cl; ++c) s += __ldcg(p.partials + ((int64_t)c * 2) * p.n + col);
        Crow[col] = read_c ? p.alpha * s + p.beta * Crow[col] : p.alpha * s;
    }
}

__device__ __forceinline__ int long_segment(int total, int long_grid) {
    const int s = (int)(((int64_t)total + long_grid - 1) / long_grid);
    return s > LONG_MIN_SEGMENT ? s : LONG_MIN_SEGMENT;
}

template <typename T, int W, int G, int R>
__global__ void __launch_bounds__(LONG_THREADS, SPMM_LONG_MIN_BLOCKS)
long_kernel(SpmmParams<T> p) {
    using C = Cfg<T, W, G, R>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* red = reinterpret_cast<T*>(smem_raw);      // [LONG_WARPS][SLOTS * W]
    wait_for_predecessor();
    const int nl = p.hdr[HDR_COUNT_LONG];
    const int total = p.hdr[HDR_LONG_NNZ];
    if (nl == 0 || total == 0) return;
    const int seg = long_segment(total, p.long_grid);
    const int s0 = (int)min((int64_t)blockIdx.x * seg, (int64_t)total);
    if (s0 >= total) return;                      // uniform per CTA
    const int s1 = (int)min((int64_t)s0 + seg, (int64_t)total);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane & (G - 1), gi = lane / G;
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
                zero_acc<T, W, R>(acc);
                accumulate_range<T, W, G, R>(acc, p, wl, wh, Bp, vbase, pw, pol_s);
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
                                              p.alpha, p.beta, read_c, p.keep_c);
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

    // Split rows.  This CTA holds a partial of r0 (slot 0) unless r0 lies wholly
    // inside its range, and of its last row (slot 1) if that row runs past the
    // range.  Each CTA sharing a row counts its partial once; the CTA whose
    // count completes the row sums every partial of it in CTA order (a fixed
    // order, whichever CTA finishes last) and applies the epilogue.
    __shared__ int s_finish[2];
    int lo1 = r0, hi1 = nl - 1;                   // last row: largest r with long_pre[r] < s1
    while (lo1 < hi1) {
        const int mid = (lo1 + hi1 + 1) >> 1;
        if (p.long_pre[mid] < s1) lo1 = mid; else hi1 = mid - 1;
    }
    const int rlast = lo1;
    __threadfence();                              // partial writes before the counters
    __syncthreads();
    if (threadIdx.x < 2) {
        const int r = threadIdx.x == 0 ? r0 : rlast;
        int fin = 0;
        if (threadIdx.x == 0 || rlast != r0) {
            const int pre_r = p.long_pre[r], pre_r1 = p.long_pre[r + 1];
            if (!(pre_r >= s0 && pre_r1 <= s1)) {
                const int cf = pre_r / seg, cl = (pre_r1 - 1) / seg;
                fin = atomicAdd(p.long_cnt + r, 1) == cl - cf;
            }
        }
        s_finish[threadIdx.x] = fin;
    }
    __syncthreads();
    for (int which = 0; which < 2; ++which) {
        if (!s_finish[which]) continue;           // uniform per CTA
        __threadfence();
        const int r = which == 0 ? r0 : rlast;
        finish_split_row<T>(p, lrows, r, seg, read_c);
        // every sharer has counted: leave the counter at zero for the next
        // product that reuses these bins (an analysed plan)
        if (threadIdx.x == 0) p.long_cnt[r] = 0;
    }
}

}  // namespace spmm
