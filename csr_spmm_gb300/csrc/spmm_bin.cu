// Row-binning pre-pass: a stable partition of the rows of A by length into
// short / medium / long lists, plus the exclusive prefix of the medium-row and
// long-row lengths (the medium prefix balances medium rows across warps by
// entries; the long prefix drives the long-row CTA split).
//
// Reads row_ptr only.  For m <= 2048 a single CTA does everything in one
// launch; otherwise two launches (three when the tiles exceed about one wave,
// m > 2.49 M, where a one-CTA scan of the tile records runs in between):
//   bin_count   per tile (512, 1024 or 2048 rows, the smallest that keeps the
//               tile count within about one wave): rows per bin, entries in
//               medium and long rows
//   bin_scatter per tile: the tile's offsets and the bin totals, reduced
//               from the tile records by each CTA (CTA 0 writes the
//               header), or read from the scan; stable ranks (warp ballots + per-warp prefix),
//               writes rowlist, med_pre and long_pre, and zeroes the
//               per-long-row counters of the long-row kernel; a tile of
//               short rows only just lists its row range
// Ranks come from ballots in ascending row order, never from atomics, so the
// lists (and everything computed from them) are identical on every call.
#include "spmm_internal.h"

namespace spmm {
namespace {

// tile record words
enum { R_SHORT = 0, R_MED = 1, R_LONG = 2, R_LONG_NNZ = 3, R_MED_NNZ = 4, R_USED = 5 };

__device__ __forceinline__ int classify(int len, int short_max, int long_min) {
    return len <= short_max ? BIN_SHORT : (len < long_min ? BIN_MEDIUM : BIN_LONG);
}

__device__ __forceinline__ int row_len(const int* row_ptr, int row, int m) {
    return row < m ? __ldg(row_ptr + row + 1) - __ldg(row_ptr + row) : -1;
}

// Per-warp totals of one tile (ITEMS rows per thread) into s_part[warp][word];
// the caller synchronises and adds the warps in order (tile_total).
template <int ITEMS>
__device__ __forceinline__ void tile_record(const int* __restrict__ row_ptr, int m, int short_max,
                                            int long_min, int tile, int (*s_part)[R_USED]) {
    int c[R_USED] = {0, 0, 0, 0, 0};
    const int base = tile * BIN_THREADS * ITEMS;
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
        const int row = base + j * BIN_THREADS + threadIdx.x;
        const int len = row_len(row_ptr, row, m);
        const int b = len >= 0 ? classify(len, short_max, long_min) : -1;
        c[R_SHORT] += b == BIN_SHORT;
        c[R_MED] += b == BIN_MEDIUM;
        c[R_LONG] += b == BIN_LONG;
        c[R_LONG_NNZ] += b == BIN_LONG ? len : 0;
        c[R_MED_NNZ] += b == BIN_MEDIUM ? len : 0;
    }
#pragma unroll
    for (int w = 0; w < R_USED; ++w)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) c[w] += __shfl_xor_sync(FULL, c[w], off);
    if ((threadIdx.x & 31) == 0)
#pragma unroll
        for (int w = 0; w < R_USED; ++w) s_part[threadIdx.x >> 5][w] = c[w];
}

__device__ __forceinline__ int tile_total(const int (*s_part)[R_USED], int word) {
    int t = 0;
#pragma unroll
    for (int w = 0; w < BIN_THREADS / 32; ++w) t += s_part[w][word];
    return t;
}

// Stable scatter of one tile.  run[] holds the tile's offsets within each bin
// (and within the medium / long length prefixes); bin_base the list offsets.
template <int ITEMS>
__device__ __forceinline__ void tile_scatter(const int* __restrict__ row_ptr, int m, int short_max,
                                             int long_min, int tile, int (&run)[R_USED],
                                             const int (&bin_base)[3], int* __restrict__ rowlist,
                                             int* __restrict__ med_pre, int* __restrict__ long_pre,
                                             int* __restrict__ long_cnt, int (*s_wc)[R_USED]) {
    constexpr int NW = BIN_THREADS / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int base = tile * BIN_THREADS * ITEMS;
    for (int j = 0; j < ITEMS; ++j) {
        const int row = base + j * BIN_THREADS + threadIdx.x;
        const int len = row_len(row_ptr, row, m);
        const int b = len >= 0 ? classify(len, short_max, long_min) : -1;
        unsigned mask[3];
        int rank[3];
#pragma unroll
        for (int c = 0; c < 3; ++c) {
            mask[c] = __ballot_sync(FULL, b == c);
            rank[c] = __popc(mask[c] & lt_mask);
        }
        // inclusive warp scans of long-row and medium-row lengths
        const int llen = b == BIN_LONG ? len : 0;
        const int mlen = b == BIN_MEDIUM ? len : 0;
        int lincl = llen, mincl = mlen;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(FULL, lincl, off);
            const int z = __shfl_up_sync(FULL, mincl, off);
            if (lane >= off) {
                lincl += y;
                mincl += z;
            }
        }
        if (lane == 31) {
            s_wc[warp][R_SHORT] = __popc(mask[0]);
            s_wc[warp][R_MED] = __popc(mask[1]);
            s_wc[warp][R_LONG] = __popc(mask[2]);
            s_wc[warp][R_LONG_NNZ] = lincl;
            s_wc[warp][R_MED_NNZ] = mincl;
        }
        __syncthreads();
        int wpre[R_USED] = {0, 0, 0, 0, 0}, tot[R_USED] = {0, 0, 0, 0, 0};
#pragma unroll
        for (int w = 0; w < NW; ++w) {
#pragma unroll
            for (int c = 0; c < R_USED; ++c) {
                const int x = s_wc[w][c];
                if (w < warp) wpre[c] += x;
                tot[c] += x;
            }
        }
        if (b >= 0) {
            const int pos_in_bin = run[b] + wpre[b] + rank[b];
            rowlist[bin_base[b] + pos_in_bin] = row;
            if (b == BIN_LONG) {
                long_pre[pos_in_bin] = run[R_LONG_NNZ] + wpre[R_LONG_NNZ] + lincl - llen;
                long_cnt[pos_in_bin] = 0;
            }
            if (b == BIN_MEDIUM) med_pre[pos_in_bin] = run[R_MED_NNZ] + wpre[R_MED_NNZ] + mincl - mlen;
        }
#pragma unroll
        for (int c = 0; c < R_USED; ++c) run[c] += tot[c];
        __syncthreads();   // s_wc is rewritten by the next sub-tile
    }
}

// A tile whose rows are all short (the count pass says so) lists them in
// order at its offset in the short bin: rowlist[off + i] = first row + i.  No
// re-read of row_ptr, no ranks, no barriers; there are no medium or long rows
// to place.  Same list as tile_scatter gives.
template <int ITEMS>
__device__ __forceinline__ void tile_all_short(int m, int tile, int short_off,
                                               int* __restrict__ rowlist) {
    const int base = tile * BIN_THREADS * ITEMS;
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
        const int i = j * BIN_THREADS + threadIdx.x;
        if (base + i < m) rowlist[short_off + i] = base + i;
    }
}

__device__ __forceinline__ void write_header(const int (&total)[R_USED], int* __restrict__ hdr,
                                             int* __restrict__ med_pre, int* __restrict__ long_pre) {
    hdr[HDR_COUNT_SHORT] = total[R_SHORT];
    hdr[HDR_COUNT_MEDIUM] = total[R_MED];
    hdr[HDR_COUNT_LONG] = total[R_LONG];
    hdr[HDR_LONG_NNZ] = total[R_LONG_NNZ];
    hdr[HDR_MED_NNZ] = total[R_MED_NNZ];
    long_pre[total[R_LONG]] = total[R_LONG_NNZ];   // closing entries of the prefixes
    med_pre[total[R_MED]] = total[R_MED_NNZ];
}

// ---- m <= BIN_SINGLE_ROWS: the whole pre-pass in one CTA ----
__global__ void __launch_bounds__(BIN_THREADS)
bin_single_kernel(const int* __restrict__ row_ptr, int m, int short_max, int long_min,
                  int* __restrict__ hdr, int* __restrict__ rowlist, int* __restrict__ med_pre,
                  int* __restrict__ long_pre, int* __restrict__ long_cnt) {
    __shared__ int s_part[BIN_THREADS / 32][R_USED];
    __shared__ int s_wc[BIN_THREADS / 32][R_USED];
    allow_successor();
    tile_record<BIN_SINGLE_ITEMS>(row_ptr, m, short_max, long_min, 0, s_part);
    __syncthreads();
    int total[R_USED];
#pragma unroll
    for (int c = 0; c < R_USED; ++c) total[c] = tile_total(s_part, c);
    if (threadIdx.x == 0) write_header(total, hdr, med_pre, long_pre);
    if (total[R_SHORT] == m) {                    // uniform: every row is short
        tile_all_short<BIN_SINGLE_ITEMS>(m, 0, 0, rowlist);
        return;
    }
    int run[R_USED] = {0, 0, 0, 0, 0};
    const int bin_base[3] = {0, total[R_SHORT], total[R_SHORT] + total[R_MED]};
    tile_scatter<BIN_SINGLE_ITEMS>(row_ptr, m, short_max, long_min, 0, run, bin_base, rowlist,
                                   med_pre, long_pre, long_cnt, s_wc);
}

// ---- many tiles ----
template <int ITEMS>
__global__ void __launch_bounds__(BIN_THREADS)
bin_count_kernel(const int* __restrict__ row_ptr, int m, int short_max, int long_min,
                 int* __restrict__ tile_counts) {
    __shared__ int s_part[BIN_THREADS / 32][R_USED];
    allow_successor();
    tile_record<ITEMS>(row_ptr, m, short_max, long_min, blockIdx.x, s_part);
    __syncthreads();
    if (threadIdx.x < BIN_REC) tile_counts[blockIdx.x * BIN_REC + threadIdx.x] =
        threadIdx.x < R_USED ? tile_total(s_part, threadIdx.x) : 0;
}

// Exclusive scan of the tile records over all tiles, by one CTA.
constexpr int SCAN_THREADS = 1024;

__global__ void __launch_bounds__(SCAN_THREADS)
bin_scan_kernel(const int* __restrict__ tile_counts, int tiles, int* __restrict__ tile_offsets,
                int* __restrict__ hdr, int* __restrict__ med_pre, int* __restrict__ long_pre) {
    __shared__ int s_warp[32][R_USED];
    __shared__ int s_carry[R_USED];
    wait_for_predecessor();
    allow_successor();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < R_USED) s_carry[threadIdx.x] = 0;
    __syncthreads();
    for (int t0 = 0; t0 < tiles; t0 += SCAN_THREADS) {
        const int t = t0 + threadIdx.x;
        int v[R_USED], incl[R_USED];
#pragma unroll
        for (int c = 0; c < R_USED; ++c) {
            v[c] = t < tiles ? tile_counts[t * BIN_REC + c] : 0;
            int x = v[c];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(FULL, x, off);
                if (lane >= off) x += y;
            }
            incl[c] = x;
            if (lane == 31) s_warp[warp][c] = x;
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int c = 0; c < R_USED; ++c) {
                int x = s_warp[lane][c];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(FULL, x, off);
                    if (lane >= off) x += y;
                }
                s_warp[lane][c] = x;   // inclusive over warps
            }
        }
        __syncthreads();
        int carry_next[R_USED];
#pragma unroll
        for (int c = 0; c < R_USED; ++c) {
            const int warp_excl = warp > 0 ? s_warp[warp - 1][c] : 0;
            if (t < tiles) tile_offsets[t * BIN_REC + c] = s_carry[c] + warp_excl + incl[c] - v[c];
            carry_next[c] = s_carry[c] + s_warp[31][c];
        }
        __syncthreads();
        if (threadIdx.x < R_USED) s_carry[threadIdx.x] = carry_next[threadIdx.x];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        int total[R_USED];
#pragma unroll
        for (int c = 0; c < R_USED; ++c) total[c] = s_carry[c];
        write_header(total, hdr, med_pre, long_pre);
    }
}

// The tile's offsets in every bin and prefix, and the bin totals.  SELF: the
// CTA reduces the tile records itself (used while there are at most
// BIN_WAVE_TILES of them, read from L2: this replaces the one-CTA scan
// launch); the records of the tiles before its own give its offsets, all of
// them the totals, and CTA 0 writes the header.  Otherwise bin_scan_kernel
// has written the offsets and the header.
template <int ITEMS, bool SELF>
__global__ void __launch_bounds__(BIN_THREADS)
bin_scatter_kernel(const int* __restrict__ row_ptr, int m, int short_max, int long_min,
                   const int* __restrict__ tile_counts, const int* __restrict__ tile_offsets,
                   int tiles, int* __restrict__ hdr, int* __restrict__ rowlist,
                   int* __restrict__ med_pre, int* __restrict__ long_pre,
                   int* __restrict__ long_cnt) {
    constexpr int NW = BIN_THREADS / 32;
    __shared__ int s_wc[NW][R_USED];
    __shared__ int s_red[NW][2 * R_USED];
    wait_for_predecessor();
    allow_successor();
    int run[R_USED], total[R_USED];
    if constexpr (SELF) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int before[R_USED] = {0, 0, 0, 0, 0}, all[R_USED] = {0, 0, 0, 0, 0};
        for (int t = threadIdx.x; t < tiles; t += BIN_THREADS) {
#pragma unroll
            for (int c = 0; c < R_USED; ++c) {
                const int v = tile_counts[t * BIN_REC + c];
                all[c] += v;
                before[c] += t < (int)blockIdx.x ? v : 0;
            }
        }
#pragma unroll
        for (int c = 0; c < R_USED; ++c)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                before[c] += __shfl_xor_sync(FULL, before[c], off);
                all[c] += __shfl_xor_sync(FULL, all[c], off);
            }
        if (lane == 0)
#pragma unroll
            for (int c = 0; c < R_USED; ++c) {
                s_red[warp][c] = before[c];
                s_red[warp][R_USED + c] = all[c];
            }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < R_USED; ++c) {
            int b = 0, a = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                b += s_red[w][c];
                a += s_red[w][R_USED + c];
            }
            run[c] = b;
            total[c] = a;
        }
        if (blockIdx.x == 0 && threadIdx.x == 0) write_header(total, hdr, med_pre, long_pre);
    } else {
#pragma unroll
        for (int c = 0; c < R_USED; ++c) run[c] = tile_offsets[blockIdx.x * BIN_REC + c];
        total[R_SHORT] = hdr[HDR_COUNT_SHORT];
        total[R_MED] = hdr[HDR_COUNT_MEDIUM];
    }
    const int rows_in_tile = min(BIN_THREADS * ITEMS, m - (int)blockIdx.x * BIN_THREADS * ITEMS);
    if (tile_counts[blockIdx.x * BIN_REC + R_SHORT] == rows_in_tile) {   // uniform per CTA
        tile_all_short<ITEMS>(m, blockIdx.x, run[R_SHORT], rowlist);
        return;
    }
    const int bin_base[3] = {0, total[R_SHORT], total[R_SHORT] + total[R_MED]};
    tile_scatter<ITEMS>(row_ptr, m, short_max, long_min, blockIdx.x, run, bin_base, rowlist,
                        med_pre, long_pre, long_cnt, s_wc);
}

}  // namespace

cudaError_t launch_binning(const int* row_ptr, int m, int short_max, int long_min,
                           const BinScratch& s, cudaStream_t st, bool overlap) {
    if (m <= 0) return cudaSuccess;
    const dim3 blk(BIN_THREADS);
    if (m <= BIN_SINGLE_ROWS)
        return launch_chained(bin_single_kernel, dim3(1), blk, 0, st, false, row_ptr, m,
                              short_max, long_min, s.hdr, s.rowlist, s.med_pre, s.long_pre,
                              s.long_cnt);
    auto count = s.items == 8 ? bin_count_kernel<8> : s.items == 4 ? bin_count_kernel<4>
                                                                      : bin_count_kernel<2>;
    cudaError_t e = launch_chained(count, dim3(s.tiles), blk, 0, st, false, row_ptr, m,
                                   short_max, long_min, s.tile_counts);
    if (e != cudaSuccess) return e;
    if (s.tiles <= BIN_WAVE_TILES) {
        auto scatter = s.items == 8 ? bin_scatter_kernel<8, true>
                       : s.items == 4 ? bin_scatter_kernel<4, true> : bin_scatter_kernel<2, true>;
        return launch_chained(scatter, dim3(s.tiles), blk, 0, st, overlap, row_ptr, m,
                              short_max, long_min, (const int*)s.tile_counts,
                              (const int*)s.tile_offsets, s.tiles, s.hdr, s.rowlist, s.med_pre,
                              s.long_pre, s.long_cnt);
    }
    e = launch_chained(bin_scan_kernel, dim3(1), dim3(SCAN_THREADS), 0, st, overlap,
                       (const int*)s.tile_counts, s.tiles, s.tile_offsets, s.hdr, s.med_pre,
                       s.long_pre);
    if (e != cudaSuccess) return e;
    auto scatter = s.items == 8 ? bin_scatter_kernel<8, false>
                   : s.items == 4 ? bin_scatter_kernel<4, false> : bin_scatter_kernel<2, false>;
    return launch_chained(scatter, dim3(s.tiles), blk, 0, st, overlap, row_ptr, m, short_max,
                          long_min, (const int*)s.tile_counts, (const int*)s.tile_offsets,
                          s.tiles, s.hdr, s.rowlist, s.med_pre, s.long_pre, s.long_cnt);
}

}  // namespace spmm
