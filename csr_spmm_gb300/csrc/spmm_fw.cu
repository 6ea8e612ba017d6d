// The Frank-Wolfe gradient scan of the SEACells B update (bixverse page,
// seacells_kernels.rs: `fw_argmin_b` and `reduce_argmin_blocks`):
//
//   G[i, c] = sum_m K2B[i, m] * t1[m, c] - T2[i, c]          (never stored)
//   min_val[c], min_idx[c] = minimum of G[:, c] and the lowest row holding it
//   gap = sum over B's stored entries of B[i, c] * G[i, c]
//
// GB300 layout: t1 (k x k, small) is expanded once into a dense, zero-padded
// row-major scratch copy, so the gradient of one row is a sparse-times-dense
// product: every K2B entry (m, v) adds v times row m of the dense t1, gathered
// as 16-byte vectors (the copy stays in L1/L2 for the k of SEACells).  A warp
// owns a row and 32 x (16 / sizeof(T)) columns of it per pass; warps take rows
// in increasing order, so a lane's strict < keeps the lowest row of its share,
// and the cross-warp reduction breaks value ties on the row index.  No float
// atomics: the result does not depend on scheduling.
#include <cfloat>

#include "spmm_device.cuh"
#include "spmm_internal.h"
#include "spmm_ops.h"

namespace spmm {
namespace {

constexpr int FW_NONE = 0x7fffffff;   // "no row yet" (loses every index tie)
#ifndef SPMM_FW_SMEM
#define SPMM_FW_SMEM 1
#endif
constexpr size_t FW_SMEM_MAX = 96 * 1024;

template <typename T> __device__ __forceinline__ T largest();
template <> __device__ __forceinline__ float largest<float>() { return FLT_MAX; }
template <> __device__ __forceinline__ double largest<double>() { return DBL_MAX; }

// Dense copy of t1, one warp per row.  Duplicates of a column are adjacent
// (columns ascend within a row), so the lane holding the first entry of each
// run of equal columns sums the run in stored order: no atomics, and the
// copy is the same on every run.
template <typename T>
__global__ void __launch_bounds__(256) fw_densify(FwParams<T> p) {
    const int m = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (m >= p.k) return;
    const int lane = threadIdx.x & 31;
    T* row = p.t1d + (int64_t)m * p.ldk;
    const int q0 = p.t1_rp[m], q1 = p.t1_rp[m + 1];
    for (int q = q0 + lane; q < q1; q += 32) {
        const int c = p.t1_ci[q];
        if (q > q0 && p.t1_ci[q - 1] == c) continue;     // not the start of its run
        T v = p.t1_v[q];
        for (int r = q + 1; r < q1 && p.t1_ci[r] == c; ++r) v += p.t1_v[r];
        row[c] = v;
    }
}

// Scatter the entries of one CSR row that fall in columns [tb, tb + TILE)
// into the warp's TILE-wide shared row `buf` (zeroed by the caller).  Columns
// ascend within the row, so duplicates sit together: the lane holding the
// first entry of a run adds the run in stored order and writes the sum once.
// No atomics, so the result is the same on every run.
template <typename T, int TILE>
__device__ __forceinline__ void scatter_row(T* buf, const int* __restrict__ ci,
                                            const T* __restrict__ v, int start, int end, int tb) {
    const int lane = threadIdx.x & 31;
    for (int q = start + lane; q < end; q += 32) {
        const int c = ci[q];
        if (c < tb || c >= tb + TILE) continue;
        if (q > start && ci[q - 1] == c) continue;        // inside a run
        T x = v[q];
        for (int r = q + 1; r < end && ci[r] == c; ++r) x += v[r];
        buf[c - tb] = x;
    }
}

// One warp per row at a time; a warp takes blocks of 32 consecutive rows
// (blocks w, w + nwarps, ...) and walks each block's rows in order, so a
// lane's strict < keeps the lowest row of its share.  The row descriptors of
// a block are loaded at once (lane r: row r), and the first chunk of the next
// row's K2B entries is loaded before the current row's gathers.
// 16-byte vector load from shared memory
template <typename T, int W>
__device__ __forceinline__ void lds_vec(const T* p, T (&v)[W]) {
    if constexpr (sizeof(T) == 4) {
        const float4 x = *reinterpret_cast<const float4*>(p);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
        const double2 x = *reinterpret_cast<const double2*>(p);
        v[0] = x.x; v[1] = x.y;
    }
}

// SMEM: the column pass's slice of the dense t1 (k rows x TILE columns) is
// copied into shared memory once per pass, and the gathers read it there.
template <typename T, bool SMEM>
__global__ void __launch_bounds__(FW_THREADS) fw_scan(FwParams<T> p) {
    constexpr int W = 16 / (int)sizeof(T);
    constexpr int TILE = fw_tile<T>();
    constexpr int U = 4;                         // gathers in flight per lane
    constexpr int WPB = FW_THREADS / 32;
    const int lane = threadIdx.x & 31;
    const int wb = threadIdx.x >> 5;
    const int gw = blockIdx.x * WPB + wb;
    const int nw = p.nwarps;
    __shared__ __align__(16) T s_row[WPB][2][TILE];      // the T2 and B entries of a row
    __shared__ T s_val[WPB][TILE];
    __shared__ int s_idx[WPB][TILE];
    extern __shared__ __align__(16) unsigned char fw_dyn[];
    T* s_t1 = reinterpret_cast<T*>(fw_dyn);              // [k][TILE] when SMEM
    T* g2 = s_row[wb][0];
    T* gb = s_row[wb][1];
    double gap = 0.0;
    for (int tb = 0; tb < p.k; tb += TILE) {
        if constexpr (SMEM) {
            const int vecs = p.k * (TILE / W);
            for (int q = threadIdx.x; q < vecs; q += FW_THREADS) {
                const int m = q / (TILE / W), c = (q % (TILE / W)) * W;
                T v[W];
                BLoad<T, W>::run(p.t1d + (int64_t)m * p.ldk + tb + c, v);
#pragma unroll
                for (int e = 0; e < W; ++e) s_t1[m * TILE + c + e] = v[e];
            }
            __syncthreads();
        }
        const int cbase = tb + lane * W;        // the lane's first column (< ldk)
        T best_v[W];
        int best_i[W];
#pragma unroll
        for (int e = 0; e < W; ++e) {
            best_v[e] = largest<T>();
            best_i[e] = FW_NONE;
        }
        const T* trow = SMEM ? s_t1 + lane * W : p.t1d + cbase;
        const int tstride = SMEM ? TILE : p.ldk;
        for (int r0 = gw * 32; r0 < p.n; r0 += nw * 32) {
            const int nr = min(32, p.n - r0);
            int a0 = 0, a1 = 0, c0 = 0, c1 = 0, b0 = 0, b1 = 0;
            if (lane < nr) {
                const int r = r0 + lane;
                a0 = p.k2b_rp[r]; a1 = p.k2b_rp[r + 1];
                c0 = p.t2_rp[r];  c1 = p.t2_rp[r + 1];
                b0 = p.b_rp[r];   b1 = p.b_rp[r + 1];
            }
            // first chunk of row 0's K2B entries
            int s0 = __shfl_sync(FULL, a0, 0), s1 = __shfl_sync(FULL, a1, 0);
            int mj = (s0 + lane < s1) ? p.k2b_ci[s0 + lane] : 0;
            T vj = (s0 + lane < s1) ? p.k2b_v[s0 + lane] : T(0);
            for (int t = 0; t < nr; ++t) {
                const int i = r0 + t;
                // next row's first chunk, in flight during this row
                const int tn = t + 1 < nr ? t + 1 : t;
                const int n0 = __shfl_sync(FULL, a0, tn), n1 = __shfl_sync(FULL, a1, tn);
                int mn = 0;
                T vn = T(0);
                if (t + 1 < nr && n0 + lane < n1) {
                    mn = p.k2b_ci[n0 + lane];
                    vn = p.k2b_v[n0 + lane];
                }
                T acc[W];
#pragma unroll
                for (int e = 0; e < W; ++e) acc[e] = T(0);
                for (int s = s0; s < s1; s += 32) {
                    if (s != s0) {                      // rows longer than one chunk
                        mj = s + lane < s1 ? p.k2b_ci[s + lane] : 0;
                        vj = s + lane < s1 ? p.k2b_v[s + lane] : T(0);
                    }
                    const int cnt = min(32, s1 - s);
                    for (int t0 = 0; t0 < cnt; t0 += U) {
                        T bv[U][W];
                        T av[U];
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            // entries past the chunk read row 0 with weight 0
                            const int m = __shfl_sync(FULL, mj, (t0 + u) & 31);
                            const T x = __shfl_sync(FULL, vj, (t0 + u) & 31);
                            av[u] = (t0 + u < cnt) ? x : T(0);
                            const T* src = trow + (int64_t)((t0 + u < cnt) ? m : 0) * tstride;
                            if constexpr (SMEM) lds_vec<T, W>(src, bv[u]);
                            else BLoad<T, W>::run(src, bv[u]);
                        }
#pragma unroll
                        for (int u = 0; u < U; ++u)
#pragma unroll
                            for (int e = 0; e < W; ++e) acc[e] = fma(av[u], bv[u][e], acc[e]);
                    }
                }
                // G = acc - T2[i, :]: scatter the row's T2 entries into shared memory
                const int u0 = __shfl_sync(FULL, c0, t), u1 = __shfl_sync(FULL, c1, t);
                const int v0 = __shfl_sync(FULL, b0, t), v1 = __shfl_sync(FULL, b1, t);
#pragma unroll
                for (int e = 0; e < W; ++e) g2[lane * W + e] = T(0);
                __syncwarp();
                scatter_row<T, TILE>(g2, p.t2_ci, p.t2_v, u0, u1, tb);
                __syncwarp();
#pragma unroll
                for (int e = 0; e < W; ++e) acc[e] -= g2[lane * W + e];
                // gap += B[i, c] * G[i, c] over B's entries (most rows hold none)
                if (v1 > v0) {
#pragma unroll
                    for (int e = 0; e < W; ++e) gb[lane * W + e] = T(0);
                    __syncwarp();
                    scatter_row<T, TILE>(gb, p.b_ci, p.b_v, v0, v1, tb);
                    __syncwarp();
#pragma unroll
                    for (int e = 0; e < W; ++e) {
                        const T b = gb[lane * W + e];
                        if (b != T(0)) gap += (double)b * (double)acc[e];
                    }
                }
                __syncwarp();                           // buffers reused by the next row
#pragma unroll
                for (int e = 0; e < W; ++e)
                    if (cbase + e < p.k && acc[e] < best_v[e]) {   // strict: lowest row kept
                        best_v[e] = acc[e];
                        best_i[e] = i;
                    }
                s0 = n0;
                s1 = n1;
                mj = mn;
                vj = vn;
            }
        }
        // the block's minima: its warps' candidates combined in warp order
#pragma unroll
        for (int e = 0; e < W; ++e) {
            s_val[wb][lane * W + e] = best_v[e];
            s_idx[wb][lane * W + e] = best_i[e];
        }
        __syncthreads();
        for (int c = threadIdx.x; c < TILE; c += FW_THREADS) {
            T bv = s_val[0][c];
            int bi = s_idx[0][c];
            for (int w = 1; w < WPB; ++w) {
                const T v = s_val[w][c];
                const int r = s_idx[w][c];
                if (v < bv || (v == bv && r < bi)) {
                    bv = v;
                    bi = r;
                }
            }
            p.part_val[(int64_t)blockIdx.x * p.ldk + tb + c] = bv;
            p.part_idx[(int64_t)blockIdx.x * p.ldk + tb + c] = bi;
        }
        __syncthreads();
    }
    // the block's gap: fixed xor tree over lanes, then warps in order
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) gap += __shfl_xor_sync(FULL, gap, off);
    __shared__ double s_gap[WPB];
    if (lane == 0) s_gap[wb] = gap;
    __syncthreads();
    if (threadIdx.x == 0) {
        double g = 0.0;
        for (int w = 0; w < WPB; ++w) g += s_gap[w];
        p.part_gap[blockIdx.x] = g;
    }
}

// Warps 0 .. k-1: one column each; lanes take blocks lane, lane + 32, ...
// and the (value, row) candidates are combined by the order "smaller value,
// then lower row", a total order, so the result does not depend on the
// combining order.  The last block sums the gap partials in a fixed order.
template <typename T>
__global__ void __launch_bounds__(256) fw_reduce(FwParams<T> p) {
    const int cblocks = (p.k + 7) / 8;
    if ((int)blockIdx.x < cblocks) {
        const int c = blockIdx.x * 8 + (threadIdx.x >> 5);
        if (c >= p.k) return;
        const int lane = threadIdx.x & 31;
        T best = largest<T>();
        int row = FW_NONE;
        for (int b = lane; b < p.nblocks; b += 32) {
            const T v = p.part_val[(int64_t)b * p.ldk + c];
            const int r = p.part_idx[(int64_t)b * p.ldk + c];
            if (v < best || (v == best && r < row)) {
                best = v;
                row = r;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const T v = __shfl_xor_sync(FULL, best, off);
            const int r = __shfl_xor_sync(FULL, row, off);
            if (v < best || (v == best && r < row)) {
                best = v;
                row = r;
            }
        }
        if (lane == 0) {
            p.out_val[c] = best;
            p.out_idx[c] = row == FW_NONE ? 0 : row;   // nothing below the start: row 0
        }
        return;
    }
    __shared__ double s[256];
    double a = 0.0;
    for (int b = threadIdx.x; b < p.nblocks; b += 256) a += p.part_gap[b];
    s[threadIdx.x] = a;
    __syncthreads();
    for (int h = 128; h > 0; h >>= 1) {
        if ((int)threadIdx.x < h) s[threadIdx.x] += s[threadIdx.x + h];
        __syncthreads();
    }
    if (threadIdx.x == 0) *p.out_gap = (T)s[0];
}

// Shared-memory bytes for the t1 slice of one column pass; 0 when it is too
// large to leave room for at least two blocks per SM (the gathers then read
// the dense copy through L1).
template <typename T>
size_t fw_smem_bytes(int k) {
    const size_t b = (size_t)k * fw_tile<T>() * sizeof(T);
    return (SPMM_FW_SMEM && b <= FW_SMEM_MAX) ? b : 0;
}

}  // namespace

template <typename T>
cudaError_t launch_fw(const FwParams<T>& p, int grid, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(p.t1d, 0, sizeof(T) * (size_t)p.k * p.ldk, st);
    if (e != cudaSuccess) return e;
    if (p.k > 0) fw_densify<T><<<(p.k + 7) / 8, 256, 0, st>>>(p);
    const size_t smem = fw_smem_bytes<T>(p.k);
    if (smem > 0) {
        e = cudaFuncSetAttribute(fw_scan<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        fw_scan<T, true><<<grid, FW_THREADS, smem, st>>>(p);
    } else {
        fw_scan<T, false><<<grid, FW_THREADS, 0, st>>>(p);
    }
    fw_reduce<T><<<(p.k + 7) / 8 + 1, 256, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename T>
int fw_blocks_per_sm(int k) {
    int b = 0;
    const size_t smem = fw_smem_bytes<T>(k);
    cudaError_t e;
    if (smem > 0) {
        e = cudaFuncSetAttribute(fw_scan<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fw_scan<T, true>, FW_THREADS,
                                                              smem);
    } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fw_scan<T, false>, FW_THREADS, 0);
    }
    if (e != cudaSuccess || b < 1) {
        cudaGetLastError();
        b = 1;
    }
    return b;
}

template cudaError_t launch_fw<float>(const FwParams<float>&, int, cudaStream_t);
template cudaError_t launch_fw<double>(const FwParams<double>&, int, cudaStream_t);
template int fw_blocks_per_sm<float>(int);
template int fw_blocks_per_sm<double>(int);

}  // namespace spmm
