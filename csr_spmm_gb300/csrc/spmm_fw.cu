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
// atomics: the result does not depend on scheduling.  Binary32 scans with
// k <= 104 take the tensor-core scan instead (fw_scan_tc, below): the same
// outputs, with the contraction K2B t1 done by tcgen05 MMAs a tile of 128
// rows at a time.
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
// binary32 scans with k <= FWTC_MAXK run on the tensor cores (fw_scan_tc)
#ifndef SPMM_FW_TC
#define SPMM_FW_TC 1
#endif

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


// ---------------------------------------------------------------------------
// Tensor-core scan (binary32, k <= FWTC_MAXK): the gradient of 128 rows at a
// time is one tile D = A t1 on the fifth-generation tensor cores, A the
// tile's K2B rows made dense (k columns) in shared memory.  Operands are
// binary32 split into two tf32 parts, x = x_hi + x_lo (each rounded to tf32,
// x - x_hi exact), and D = A_hi t1_hi + A_hi t1_lo + A_lo t1_hi: three
// kind::tf32 MMAs per 8-wide k step, each product of tf32 parts exact in
// binary32, the dropped A_lo t1_lo and rounding residues below 2^-21 of
// |a||t|, with binary32 accumulation in tensor memory.  One thread issues
// the MMAs; completion is signalled on an mbarrier; the 128 x N accumulator
// is read back with tcgen05.ld (warp w: lanes 32 (w % 4) .. + 31, one row
// per thread, column chunks by w / 4) into a shared-memory tile where T2 is
// subtracted (duplicate columns summed in stored order first, as in the
// CUDA-core scan), B's entries add to the gap, and four groups of threads
// keep each column's minimum over 32-row slices of the block's rows in
// ascending order (strict <: lowest row), combined at the end by value,
// then row.  While the MMAs run, the tile's T2 rows, the next tile's K2B
// rows and the tile's B entries are loaded.  Operand layout:
// K-major, no swizzle, 8-row x 16-byte core matrices; within an 8-row group
// the k direction's core matrices are 128 bytes apart (the descriptor's
// leading byte offset), and the groups kp * 32 bytes apart (stride offset).
constexpr int FWTC_THREADS = 512;
constexpr int FWTC_M = 128;                      // rows per tile: the MMA's M
constexpr int FWTC_MAXK = 104;
constexpr int FWTC_WAIT_LIMIT = 1 << 24;

struct FwTcGeo {
    int kp;             // k rounded up to the MMA's k step (8)
    int nn;             // N of the MMA: k rounded up to 16
    int tcols;          // tensor-memory columns (a power of two, >= 32)
    int gstride;        // row stride of the gradient tile (floats)
    size_t a_bytes;     // one A part (128 x kp)
    size_t b_bytes;     // one t1 part (nn x kp)
    size_t region_a;    // both A parts, or the gradient tile, whichever is larger
    size_t smem;        // dynamic shared memory
};

__host__ __device__ inline FwTcGeo fwtc_geo(int k) {
    FwTcGeo g;
    g.kp = (k + 7) / 8 * 8;
    g.nn = (k + 15) / 16 * 16;
    g.tcols = 32;
    while (g.tcols < g.nn) g.tcols *= 2;
    g.gstride = g.nn + 1;
    g.a_bytes = (size_t)(FWTC_M / 8) * g.kp * 32;
    g.b_bytes = (size_t)(g.nn / 8) * g.kp * 32;
    const size_t gt = (size_t)FWTC_M * g.gstride * sizeof(float);
    g.region_a = ((2 * g.a_bytes > gt ? 2 * g.a_bytes : gt) + 127) / 128 * 128;
    g.smem = g.region_a + 2 * g.b_bytes;
    return g;
}

inline bool fw_tc_ok(int k) {
    return SPMM_FW_TC && k >= 1 && k <= FWTC_MAXK && fwtc_geo(k).smem <= 200 * 1024;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
// shared-memory matrix descriptor: start, leading and stride byte offsets
// (all in 16-byte units), descriptor version 1, no swizzle
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
__device__ __forceinline__ int kmajor_off(int r, int kk, int kp) {
    return (r >> 3) * (kp * 32) + (kk >> 2) * 128 + (r & 7) * 16 + (kk & 3) * 4;
}
__device__ __forceinline__ void split_tf32(float v, float& hi, float& lo) {
    uint32_t h, l;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(v));
    hi = __uint_as_float(h);
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(l) : "f"(v - hi));
    lo = __uint_as_float(l);
}
__device__ __forceinline__ void umma_tf32(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          int accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// The rows of a tile that one warp handles: tile rows 8 w .. 8 w + 7, four
// lanes per row (lane l: row l / 4, entries l % 4, l % 4 + 4, ...), so that
// the lanes of one store cover eight consecutive rows, whose 16-byte core
// matrix rows lie in different shared-memory banks.  The first FWTC_STEPS
// steps (4 entries of each row per step) are loaded ahead of their use,
// while the MMAs run.
constexpr int FWTC_WARPS = FWTC_THREADS / 32;
constexpr int FWTC_STEPS = 8;
static_assert(FWTC_M == FWTC_WARPS * 8, "eight rows per warp");
struct FwRows {
    int s, e;                                    // this lane's row: entries [s, e)
    int c[FWTC_STEPS];
    float v[FWTC_STEPS];
};

__device__ __forceinline__ void fw_rows_extents(FwRows& R, const int* __restrict__ rp, int r0,
                                                int nr) {
    const int r = (int)(threadIdx.x >> 5) * 8 + (int)((threadIdx.x & 31) >> 2);
    R.s = 0;
    R.e = 0;
    if (r < nr) {
        R.s = rp[r0 + r];
        R.e = rp[r0 + r + 1];
    }
}

__device__ __forceinline__ void fw_rows_entries(FwRows& R, const int* __restrict__ ci,
                                                const float* __restrict__ val) {
    const int sub = threadIdx.x & 3;
#pragma unroll
    for (int t = 0; t < FWTC_STEPS; ++t) {
        const int q = R.s + 4 * t + sub;
        R.c[t] = q < R.e ? ci[q] : -1;
        R.v[t] = q < R.e ? val[q] : 0.f;
    }
}

// Every run of equal columns in the warp's rows: f(row in tile, column, sum
// of the run in stored order), called by the lane holding the run's first
// entry.  Neighbouring entries of a row sit in neighbouring lanes of its
// four; longer rows load their further steps here.  No block barrier: each
// warp touches only its own rows.
template <typename F>
__device__ __forceinline__ void fw_rows_apply(const FwRows& R, const int* __restrict__ ci,
                                              const float* __restrict__ val, F f) {
    const int lane = threadIdx.x & 31, sub = lane & 3, g0 = lane & ~3;
    const int r = (int)(threadIdx.x >> 5) * 8 + (lane >> 2);
    const int steps = (__reduce_max_sync(FULL, (unsigned)(R.e - R.s)) + 3) / 4;
    int last = -2;                               // the row's previous step's last column
#pragma unroll
    for (int t = 0; t < FWTC_STEPS; ++t) {
        if (t < steps) {                         // warp-uniform
            const int q = R.s + 4 * t + sub;
            const int c = R.c[t];
            int prev = __shfl_up_sync(FULL, c, 1);
            if (sub == 0) prev = last;
            int next = __shfl_down_sync(FULL, c, 1);
            const int first_next =
                t + 1 < FWTC_STEPS ? __shfl_sync(FULL, R.c[(t + 1) % FWTC_STEPS], g0) : -2;
            last = __shfl_sync(FULL, c, g0 + 3);
            if (sub == 3) next = t + 1 < FWTC_STEPS ? first_next : (q + 1 < R.e ? ci[q + 1] : -2);
            if (q < R.e && !(q > R.s && prev == c)) {
                float sum = R.v[t];
                if (q + 1 < R.e && next == c)    // a run: sum it in order
                    for (int q2 = q + 1; q2 < R.e && ci[q2] == c; ++q2) sum += val[q2];
                f(r, c, sum);
            }
        }
    }
    // rows longer than the prefetched steps
    for (int t = FWTC_STEPS; t < steps; ++t) {
        const int q = R.s + 4 * t + sub;
        const int c = q < R.e ? ci[q] : -1;
        int prev = __shfl_up_sync(FULL, c, 1);
        if (sub == 0) prev = last;
        int next = __shfl_down_sync(FULL, c, 1);
        last = __shfl_sync(FULL, c, g0 + 3);
        if (sub == 3) next = q + 1 < R.e ? ci[q + 1] : -2;
        if (q < R.e && !(q > R.s && prev == c)) {
            float sum = val[q];
            if (q + 1 < R.e && next == c)
                for (int q2 = q + 1; q2 < R.e && ci[q2] == c; ++q2) sum += val[q2];
            f(r, c, sum);
        }
    }
}

// The same walk over entries read through col(q) and val(q) (B's entries,
// staged in shared memory while the MMAs run).
constexpr int FWTC_BSTAGE = 512;                 // B entries of a tile staged at most
template <typename C, typename V, typename F>
__device__ __forceinline__ void fw_rows_apply_by(const FwRows& R, C col, V valf, F f) {
    const int lane = threadIdx.x & 31, sub = lane & 3, g0 = lane & ~3;
    const int r = (int)(threadIdx.x >> 5) * 8 + (lane >> 2);
    const int steps = (__reduce_max_sync(FULL, (unsigned)(R.e - R.s)) + 3) / 4;
    int last = -2;
    for (int t = 0; t < steps; ++t) {
        const int q = R.s + 4 * t + sub;
        const int c = q < R.e ? col(q) : -1;
        int prev = __shfl_up_sync(FULL, c, 1);
        if (sub == 0) prev = last;
        int next = __shfl_down_sync(FULL, c, 1);
        last = __shfl_sync(FULL, c, g0 + 3);
        if (sub == 3) next = q + 1 < R.e ? col(q + 1) : -2;
        if (q < R.e && !(q > R.s && prev == c)) {
            float sum = valf(q);
            if (q + 1 < R.e && next == c)
                for (int q2 = q + 1; q2 < R.e && col(q2) == c; ++q2) sum += valf(q2);
            f(r, c, sum);
        }
    }
}

__global__ void __launch_bounds__(FWTC_THREADS, 1) fw_scan_tc(FwParams<float> p) {
    extern __shared__ __align__(1024) unsigned char tc_smem[];
    __shared__ __align__(8) uint64_t s_mbar;
    __shared__ uint32_t s_tmem;
    __shared__ float s_bv[FWTC_THREADS];
    __shared__ int s_bi[FWTC_THREADS];
    __shared__ double s_gap[FWTC_WARPS];
    __shared__ int s_bcol[FWTC_BSTAGE];          // the tile's B entries, staged
    __shared__ float s_bval[FWTC_BSTAGE];
    const FwTcGeo g = fwtc_geo(p.k);
    unsigned char* sAh = tc_smem;
    unsigned char* sAl = tc_smem + g.a_bytes;
    unsigned char* sBh = tc_smem + g.region_a;
    unsigned char* sBl = sBh + g.b_bytes;
    float* sG = reinterpret_cast<float*>(tc_smem);   // after the MMAs: the gradient tile
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr(&s_tmem)), "r"(g.tcols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&s_mbar)));
    // t1 as the MMA's B operand (N x kp, K-major: B[c][m] = t1[m][c]), split;
    // consecutive threads read consecutive columns of a t1 row
#pragma unroll 4
    for (int i = tid; i < g.nn * g.kp; i += FWTC_THREADS) {
        const int m = i / g.nn, c = i - m * g.nn;
        const float v = (c < p.k && m < p.k) ? p.t1d[(int64_t)m * p.ldk + c] : 0.f;
        float hi, lo;
        split_tf32(v, hi, lo);
        const int off = kmajor_off(c, m, g.kp);
        *reinterpret_cast<float*>(sBh + off) = hi;
        *reinterpret_cast<float*>(sBl + off) = lo;
    }
    const int ntiles = (p.n + FWTC_M - 1) / FWTC_M;
    FwRows kr, tr;
    if ((int)blockIdx.x < ntiles) {
        const int r0 = blockIdx.x * FWTC_M;
        fw_rows_extents(kr, p.k2b_rp, r0, min(FWTC_M, p.n - r0));
        fw_rows_entries(kr, p.k2b_ci, p.k2b_v);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;
    const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(g.nn >> 3) << 17) |
                           ((uint32_t)(FWTC_M >> 4) << 24);
    const uint32_t sbo = (uint32_t)g.kp * 32;

    // column tid % 128 over rows 32 (tid / 128) .. + 31 of every tile
    const int mcol = tid & (FWTC_M - 1), mgrp = tid / FWTC_M;
    float best_v = FLT_MAX;
    int best_i = FW_NONE;
    double gap = 0.0;
    bool ok = true;
    int iter = 0;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++iter) {
        const int r0 = tile * FWTC_M, nr = min(FWTC_M, p.n - r0);
        // the row extents that the loads during the MMAs need, requested now
        // so that they have arrived by then: this tile's T2 and B rows, the
        // next tile's K2B rows
        FwRows br, nk;
        const int next = tile + gridDim.x;
        fw_rows_extents(tr, p.t2_rp, r0, nr);
        fw_rows_extents(br, p.b_rp, r0, nr);
        if (next < ntiles)
            fw_rows_extents(nk, p.k2b_rp, next * FWTC_M, min(FWTC_M, p.n - next * FWTC_M));
        const int b0 = p.b_rp[r0], b1 = p.b_rp[r0 + nr];
        for (size_t i = tid; i < 2 * g.a_bytes / 16; i += FWTC_THREADS)
            reinterpret_cast<float4*>(tc_smem)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncthreads();
        // the tile's K2B rows, dense and split (a run of equal columns summed
        // in stored order by the lane holding its first entry)
        fw_rows_apply(kr, p.k2b_ci, p.k2b_v, [&](int r, int c, float v) {
            if (c < 0 || c >= p.k) return;
            float hi, lo;
            split_tf32(v, hi, lo);
            const int off = kmajor_off(r, c, g.kp);
            *reinterpret_cast<float*>(sAh + off) = hi;
            *reinterpret_cast<float*>(sAl + off) = lo;
        });
        // the operands' generic-proxy stores, visible to the tensor cores
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (tid == 0) {
            const uint32_t ah = smem_addr(sAh), al = smem_addr(sAl);
            const uint32_t bh = smem_addr(sBh), bl = smem_addr(sBl);
            // a k step moves each descriptor's start by 256 bytes (16 units)
            const uint64_t dah = umma_desc(ah, 128, sbo), dal = umma_desc(al, 128, sbo);
            const uint64_t dbh = umma_desc(bh, 128, sbo), dbl = umma_desc(bl, 128, sbo);
            for (int s = 0; s < g.kp / 8; ++s) {
                const uint64_t ko = (uint64_t)s * 16;
                umma_tf32(tmem, dah + ko, dbh + ko, idesc, s > 0);
                umma_tf32(tmem, dah + ko, dbl + ko, idesc, 1);
                umma_tf32(tmem, dal + ko, dbh + ko, idesc, 1);
            }
            asm volatile(
                "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                ::"r"(smem_addr(&s_mbar)) : "memory");
        }
        // while the MMAs run: this tile's T2 rows, the next tile's K2B rows,
        // and this tile's B entries into shared memory
        fw_rows_entries(tr, p.t2_ci, p.t2_v);
        if (next < ntiles) {
            kr.s = nk.s;
            kr.e = nk.e;
            fw_rows_entries(kr, p.k2b_ci, p.k2b_v);
        }
        const bool bstaged = b1 - b0 <= FWTC_BSTAGE;
        if (bstaged && b0 + tid < b1) {
            s_bcol[tid] = p.b_ci[b0 + tid];
            s_bval[tid] = p.b_v[b0 + tid];
        }
        // the MMAs' completion (phase iter & 1), bounded
        uint32_t done = 0;
        for (int it = 0; it < FWTC_WAIT_LIMIT && !done; ++it) {
            asm volatile(
                "{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n"
                " selp.u32 %0, 1, 0, q;\n}\n"
                : "=r"(done) : "r"(smem_addr(&s_mbar)), "r"((uint32_t)(iter & 1)) : "memory");
        }
        ok = __syncthreads_and(done != 0);
        if (!ok) {
            // the MMAs may still be running: wait once more (bounded) before
            // the tensor memory is freed below
            for (int it = 0; it < FWTC_WAIT_LIMIT && !done; ++it) {
                asm volatile(
                    "{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n"
                    " selp.u32 %0, 1, 0, q;\n}\n"
                    : "=r"(done) : "r"(smem_addr(&s_mbar)), "r"((uint32_t)(iter & 1)) : "memory");
            }
            __syncthreads();
            break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // accumulator -> gradient tile: warp w reads lanes 32 (w % 4) .. + 31
        // (one row per thread), column chunks w / 4, w / 4 + 4, ...
        {
            const int quarter = warp & 3, row = quarter * 32 + lane;
            for (int c0 = (warp >> 2) * 16; c0 < g.nn; c0 += (FWTC_THREADS / 128) * 16) {
                uint32_t v[16];
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0;
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                    "%12,%13,%14,%15}, [%16];"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                      "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                      "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                    : "r"(taddr));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int j = 0; j < 16; ++j) sG[row * g.gstride + c0 + j] = __uint_as_float(v[j]);
            }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        // G = D - T2 on this warp's rows (runs of equal columns summed first),
        // then gap += B[i, c] * G[i, c] over B's entries of the same rows
        fw_rows_apply(tr, p.t2_ci, p.t2_v, [&](int r, int c, float v) {
            if (c >= 0 && c < p.k) sG[r * g.gstride + c] -= v;
        });
        __syncwarp();
        if (__any_sync(FULL, br.e > br.s)) {     // most rows of B are empty
            const auto gap_add = [&](int r, int c, float bv) {
                if (c >= 0 && c < p.k && bv != 0.f)
                    gap += (double)bv * (double)sG[r * g.gstride + c];
            };
            if (bstaged)
                fw_rows_apply_by(br, [&](int q) { return s_bcol[q - b0]; },
                                 [&](int q) { return s_bval[q - b0]; }, gap_add);
            else
                fw_rows_apply_by(br, [&](int q) { return p.b_ci[q]; },
                                 [&](int q) { return p.b_v[q]; }, gap_add);
        }
        __syncthreads();
        // column mcol's minimum over rows 32 mgrp .. + 31 of the tile, ascending
        if (mcol < p.k) {
            const int ra = mgrp * 32, rb = min(nr, ra + 32);
            if (rb - ra == 32) {                 // a full slice: loads first, compares in order
                float vs[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) vs[j] = sG[(ra + j) * g.gstride + mcol];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (vs[j] < best_v) {
                        best_v = vs[j];
                        best_i = r0 + ra + j;
                    }
            } else {
                for (int r = ra; r < rb; ++r) {
                    const float v = sG[r * g.gstride + mcol];
                    if (v < best_v) {
                        best_v = v;
                        best_i = r0 + r;
                    }
                }
            }
        }
        __syncthreads();                         // the tile is read before the next overwrites it
    }
    // each column's four candidates (value, then lower row: a total order)
    s_bv[tid] = best_v;
    s_bi[tid] = best_i;
    __syncthreads();
    if (tid < p.k) {
        float bv = s_bv[tid];
        int bi = s_bi[tid];
        for (int q = 1; q < FWTC_THREADS / FWTC_M; ++q) {
            const float v = s_bv[q * FWTC_M + tid];
            const int r = s_bi[q * FWTC_M + tid];
            if (v < bv || (v == bv && r < bi)) {
                bv = v;
                bi = r;
            }
        }
        best_v = bv;
        best_i = bi;
    }
    if (tid < p.k) {
        p.part_val[(int64_t)blockIdx.x * p.ldk + tid] = best_v;
        p.part_idx[(int64_t)blockIdx.x * p.ldk + tid] = best_i;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) gap += __shfl_xor_sync(FULL, gap, off);
    if (lane == 0) s_gap[warp] = gap;
    __syncthreads();
    if (tid == 0) {
        double t = 0.0;
        for (int w = 0; w < FWTC_WARPS; ++w) t += s_gap[w];
        // a wait that ran out leaves the gap not a number (every wait is bounded)
        p.part_gap[blockIdx.x] = ok ? t : __longlong_as_double(0x7ff8000000000000LL);
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem), "r"(g.tcols));
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
    if constexpr (sizeof(T) == 4) {
        if (fw_tc_ok(p.k)) {
            const FwTcGeo g = fwtc_geo(p.k);
            e = cudaFuncSetAttribute(fw_scan_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)g.smem);
            if (e != cudaSuccess) return e;
            fw_scan_tc<<<grid, FWTC_THREADS, g.smem, st>>>(p);
            fw_reduce<T><<<(p.k + 7) / 8 + 1, 256, 0, st>>>(p);
            return cudaGetLastError();
        }
    }
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
    if (sizeof(T) == 4 && fw_tc_ok(k)) return 1;   // the tensor-core scan: one block per SM
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
