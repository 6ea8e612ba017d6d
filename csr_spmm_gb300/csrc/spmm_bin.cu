// Row-binning pre-pass: a stable partition of the rows of A by length into
// short / medium / long lists, plus the exclusive prefix of long-row lengths
// that the long-row CTA split works from.
//
// Three launches, all reading row_ptr only:
//   bin_count   per 2048-row tile: rows per bin and entries in long rows
//   bin_scan    one CTA: exclusive scans of the tile counts, bin totals
//   bin_scatter per tile: stable ranks (warp ballots + per-warp prefix),
//               writes rowlist and long_pre
// Ranks come from ballots in ascending row order, never from atomics, so the
// lists (and everything computed from them) are identical on every call.
#include "spmm_internal.h"

namespace spmm {
namespace {

__device__ __forceinline__ int classify(int len, int short_max, int long_min) {
    return len <= short_max ? BIN_SHORT : (len < long_min ? BIN_MEDIUM : BIN_LONG);
}

__device__ __forceinline__ int row_len(const int* row_ptr, int row, int m) {
    return row < m ? __ldg(row_ptr + row + 1) - __ldg(row_ptr + row) : -1;
}

__global__ void __launch_bounds__(BIN_THREADS)
bin_count_kernel(const int* __restrict__ row_ptr, int m, int short_max, int long_min,
                 int* __restrict__ tile_counts) {
    __shared__ int s_cnt[4];
    if (threadIdx.x < 4) s_cnt[threadIdx.x] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    int c[3] = {0, 0, 0};
    int long_nnz = 0;
    const int base = blockIdx.x * BIN_TILE;
#pragma unroll
    for (int j = 0; j < BIN_ITEMS; ++j) {
        const int row = base + j * BIN_THREADS + threadIdx.x;
        const int len = row_len(row_ptr, row, m);
        if (len >= 0) {
            const int b = classify(len, short_max, long_min);
            c[b] += 1;
            if (b == BIN_LONG) long_nnz += len;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        c[0] += __shfl_xor_sync(FULL, c[0], off);
        c[1] += __shfl_xor_sync(FULL, c[1], off);
        c[2] += __shfl_xor_sync(FULL, c[2], off);
        long_nnz += __shfl_xor_sync(FULL, long_nnz, off);
    }
    if (lane == 0) {
        atomicAdd(&s_cnt[0], c[0]);   // integer counts: order-independent
        atomicAdd(&s_cnt[1], c[1]);
        atomicAdd(&s_cnt[2], c[2]);
        atomicAdd(&s_cnt[3], long_nnz);
    }
    __syncthreads();
    if (threadIdx.x < 4) tile_counts[blockIdx.x * 4 + threadIdx.x] = s_cnt[threadIdx.x];
}

// Exclusive scan of the 4-word tile records over all tiles, by one CTA.
constexpr int SCAN_THREADS = 1024;

__global__ void __launch_bounds__(SCAN_THREADS)
bin_scan_kernel(const int* __restrict__ tile_counts, int tiles, int* __restrict__ tile_offsets,
                int* __restrict__ hdr, int* __restrict__ long_pre) {
    __shared__ int s_warp[32][4];
    __shared__ int s_carry[4];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < 4) s_carry[threadIdx.x] = 0;
    __syncthreads();
    for (int t0 = 0; t0 < tiles; t0 += SCAN_THREADS) {
        const int t = t0 + threadIdx.x;
        int v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = t < tiles ? tile_counts[t * 4 + c] : 0;
        int incl[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            int x = v[c];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int y = __shfl_up_sync(FULL, x, off);
                if (lane >= off) x += y;
            }
            incl[c] = x;
            if (lane == 31) s_warp[warp][c] = x;
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                int x = s_warp[lane][c];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    int y = __shfl_up_sync(FULL, x, off);
                    if (lane >= off) x += y;
                }
                s_warp[lane][c] = x;   // inclusive over warps
            }
        }
        __syncthreads();
        int carry_next[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int warp_excl = warp > 0 ? s_warp[warp - 1][c] : 0;
            const int excl = s_carry[c] + warp_excl + incl[c] - v[c];
            if (t < tiles) tile_offsets[t * 4 + c] = excl;
            carry_next[c] = s_carry[c] + s_warp[31][c];
        }
        __syncthreads();
        if (threadIdx.x < 4) s_carry[threadIdx.x] = carry_next[threadIdx.x];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        hdr[HDR_COUNT_SHORT] = s_carry[0];
        hdr[HDR_COUNT_MEDIUM] = s_carry[1];
        hdr[HDR_COUNT_LONG] = s_carry[2];
        hdr[HDR_LONG_NNZ] = s_carry[3];
        long_pre[s_carry[2]] = s_carry[3];     // closing entry of the prefix
    }
}

__global__ void __launch_bounds__(BIN_THREADS)
bin_scatter_kernel(const int* __restrict__ row_ptr, int m, int short_max, int long_min,
                   const int* __restrict__ tile_offsets, const int* __restrict__ hdr,
                   int* __restrict__ rowlist, int* __restrict__ long_pre) {
    constexpr int NW = BIN_THREADS / 32;
    __shared__ int s_wc[NW][4];            // per warp: counts of the 3 bins + long nnz
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int base = blockIdx.x * BIN_TILE;
    int run[4];                            // running tile-local offsets
#pragma unroll
    for (int c = 0; c < 4; ++c) run[c] = tile_offsets[blockIdx.x * 4 + c];
    const int bin_base[3] = {0, hdr[HDR_COUNT_SHORT], hdr[HDR_COUNT_SHORT] + hdr[HDR_COUNT_MEDIUM]};

    for (int j = 0; j < BIN_ITEMS; ++j) {
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
        // inclusive warp scan of long-row lengths
        const int llen = b == BIN_LONG ? len : 0;
        int lincl = llen;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(FULL, lincl, off);
            if (lane >= off) lincl += y;
        }
        if (lane == 31) {
            s_wc[warp][0] = __popc(mask[0]);
            s_wc[warp][1] = __popc(mask[1]);
            s_wc[warp][2] = __popc(mask[2]);
            s_wc[warp][3] = lincl;
        }
        __syncthreads();
        int wpre[4] = {0, 0, 0, 0}, tot[4] = {0, 0, 0, 0};
#pragma unroll
        for (int w = 0; w < NW; ++w) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int x = s_wc[w][c];
                if (w < warp) wpre[c] += x;
                tot[c] += x;
            }
        }
        if (b >= 0) {
            const int pos_in_bin = run[b] + wpre[b] + rank[b];
            rowlist[bin_base[b] + pos_in_bin] = row;
            if (b == BIN_LONG) long_pre[pos_in_bin] = run[3] + wpre[3] + lincl - llen;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) run[c] += tot[c];
        __syncthreads();   // s_wc is rewritten by the next sub-tile
    }
}

}  // namespace

cudaError_t launch_binning(const int* row_ptr, int m, int short_max, int long_min,
                           const BinScratch& s, cudaStream_t st) {
    if (m <= 0) return cudaSuccess;
    bin_count_kernel<<<s.tiles, BIN_THREADS, 0, st>>>(row_ptr, m, short_max, long_min,
                                                      s.tile_counts);
    bin_scan_kernel<<<1, SCAN_THREADS, 0, st>>>(s.tile_counts, s.tiles, s.tile_offsets, s.hdr,
                                                s.long_pre);
    bin_scatter_kernel<<<s.tiles, BIN_THREADS, 0, st>>>(row_ptr, m, short_max, long_min,
                                                        s.tile_offsets, s.hdr, s.rowlist,
                                                        s.long_pre);
    return cudaGetLastError();
}

}  // namespace spmm
