// ILU(0), the incomplete LU factorisation with zero fill-in of the oxicuda
// preconditioner page (preconditioner/ilu0.rs: module doc and
// `factor_row_host`), factored in place on A's CSR values.
//
// The page analyses dependency levels on the host and launches one kernel
// per level, synchronising the stream and reading a status word back between
// levels.  Here the schedule is dataflow, on the device, without host
// round trips:
//   1. every row counts its lower entries (the rows it waits for) and adds
//      itself to the dependent count of each of them; rows with none are
//      queued; for each lower entry (i, k) it records where row k keeps its
//      pivot and where row k ends;
//   2. a prefix sum (three launches over tiles) turns the dependent counts
//      into list offsets;
//   3. the dependent lists are filled (the transpose of the strict lower
//      pattern);
//   4. one persistent launch: a warp takes the next queue slot, waits for it
//      to be filled, factors that row, publishes its final values, and
//      counts down each dependent, queueing the one whose count reaches zero.
// The counts only schedule (relaxed atomics, no fences).  The values travel
// through a separate array of published values, filled with a sentinel bit
// pattern (a signalling NaN that no arithmetic produces) before the launch:
// a row reads its pivot rows' published values and waits while one is still
// the sentinel.  Each published value is written once, by its own row, so a
// value that is not the sentinel is the final one.  A row whose final value
// is the sentinel's bit pattern itself (only an input value passed through
// unchanged can be) also sets a done flag with a release store, and a reader
// that has seen the sentinel for a while acquires that flag and takes the
// value as it is.
// Any row may run as soon as its last dependency is final, so the whole
// width of every level (the anti-diagonals of a grid) runs at once.  Waits
// are bounded, and a failure (zero or missing pivot, or a wait that ran out)
// stops every warp through a shared abort word and is reported in the status
// word.
//
// Arithmetic follows the page step for step: per lower entry k of row i in
// CSR order, ratio = a_ik / a_kk (rounded divide), stored, then for each
// j > k of row k present in row i, a_ij = a_ij - ratio * a_kj with a rounded
// multiply and a rounded subtract (no fused multiply-add), so the factors
// equal the host reference bit for bit, whatever order the rows run in.
#include <algorithm>
#include <climits>

#include "spmm_internal.h"
#include "spmm_ops.h"

namespace spmm {
namespace {

constexpr int ILU0_SINGULAR = 1;
constexpr int ILU0_WAIT_TIMEOUT = 2;
// Polls of one queue slot with no row finished anywhere before a wait gives
// up (about a second at the default).
#ifndef SPMM_ILU0_SPIN_LIMIT
#define SPMM_ILU0_SPIN_LIMIT (1 << 22)
#endif
constexpr int ILU0_SPIN_LIMIT = SPMM_ILU0_SPIN_LIMIT;
// Test builds only (0 in the library): the last row gets one extra pending
// dependency that no row counts down, so it is never queued and the waits for
// it run out.  This reaches the wait-timeout status with valid input and no
// fault: every other row is factored, the waits end by their limit, and the
// kernel returns.
#ifndef SPMM_ILU0_TEST_WITHHOLD_LAST_ROW
#define SPMM_ILU0_TEST_WITHHOLD_LAST_ROW 0
#endif
#ifndef SPMM_ILU0_SLEEP_NS
#define SPMM_ILU0_SLEEP_NS 256         // between polls of an empty queue slot
#endif
#ifndef SPMM_ILU0_POLL_EVERY
#define SPMM_ILU0_POLL_EVERY 16        // a power of two
#endif
// Fetch the structure records of a row's first two dependents while it is
// factored (0: each row's record is read when the row starts).
#ifndef SPMM_ILU0_PREFETCH
#define SPMM_ILU0_PREFETCH 1
#endif
#ifndef SPMM_ILU0_BLOCKS_PER_SM
#define SPMM_ILU0_BLOCKS_PER_SM 1      // 0: as many as fit (measured slower: idle warps poll)
#endif

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_relaxed(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// The sentinel of the published values: signalling NaNs (quiet bit clear),
// which no floating-point operation returns.
constexpr unsigned long long ILU0_SENTINEL64 = 0x7FF4C0DE5A5A5A5AULL;
constexpr unsigned ILU0_SENTINEL32 = 0x7FA5C0DEu;
__device__ __forceinline__ bool is_sentinel(double x) {
    return (unsigned long long)__double_as_longlong(x) == ILU0_SENTINEL64;
}
__device__ __forceinline__ bool is_sentinel(float x) {
    return (unsigned)__float_as_uint(x) == ILU0_SENTINEL32;
}
__device__ __forceinline__ void set_sentinel(double* q) {
    *q = __longlong_as_double((long long)ILU0_SENTINEL64);
}
__device__ __forceinline__ void set_sentinel(float* q) { *q = __uint_as_float(ILU0_SENTINEL32); }
__device__ __forceinline__ double ld_relaxed(const double* p) {
    double v;
    asm volatile("ld.relaxed.gpu.global.f64 %0, [%1];" : "=d"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float ld_relaxed(const float* p) {
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(double* p, double v) {
    asm volatile("st.relaxed.gpu.global.f64 [%0], %1;" ::"l"(p), "d"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed(float* p, float v) {
    asm volatile("st.relaxed.gpu.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed(int* p, int v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float div_rn(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ double div_rn(double a, double b) { return __ddiv_rn(a, b); }
__device__ __forceinline__ float mul_rn(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ double mul_rn(double a, double b) { return __dmul_rn(a, b); }
__device__ __forceinline__ float sub_rn(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ double sub_rn(double a, double b) { return __dsub_rn(a, b); }

// 1. lower entries per row, dependents per row, the first ready rows; and
//    for each lower entry (i, k) where row k keeps its pivot a_kk and where
//    it ends (structure only: the factorisation then needs no search)
template <typename T>
__global__ void __launch_bounds__(256) ilu0_count(Ilu0Params<T> p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    // the row's level starts as -1 (its published values: ilu0_records)
    p.done[i] = 0;
    if (p.depth) p.depth[i] = -1;
    int lower = 0;
    for (int q = p.rp[i]; q < p.rp[i + 1]; ++q) {
        const int k = p.ci[q];
        if (k >= i) break;                      // columns ascend
        atomicAdd(p.cnt + k, 1);
        ++lower;
        const int ks = p.rp[k], ke = p.rp[k + 1];
        int dp = -1;                            // first position of column k in row k
        for (int r = ks; r < ke; ++r)
            if (p.ci[r] == k) {
                dp = r;
                break;
            }
        p.piv[q] = make_int2(dp, ke);
    }
    const int withheld = (SPMM_ILU0_TEST_WITHHOLD_LAST_ROW && i == p.n - 1) ? 1 : 0;
    p.pending[i] = lower + withheld;
    if (lower + withheld == 0) p.queue[atomicAdd(p.tail, 1)] = i;
}

// 2. exclusive prefix sum of cnt into dep_ptr, then cnt is cleared to serve
//    as the fill cursor.  Three launches over tiles of ILU0_SCAN_TILE rows
//    (coalesced, every SM busy): the tiles' sums, one block scanning those
//    sums, then each tile's own scan plus its offset.
constexpr int ILU0_SCAN_TILE = 1024;

// Inclusive scan of v over a 1024-thread block; s_w holds 32 ints.
__device__ __forceinline__ int block_inclusive_scan_1024(int v, int* s_w) {
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(FULL, x, off);
        if (lane >= off) x += y;
    }
    __syncthreads();                                   // s_w free from an earlier use
    if (lane == 31) s_w[wib] = x;
    __syncthreads();
    if (wib == 0) {
        int w = s_w[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(FULL, w, off);
            if (lane >= off) w += y;
        }
        s_w[lane] = w;                                 // inclusive over the warps
    }
    __syncthreads();
    return x + (wib > 0 ? s_w[wib - 1] : 0);
}

template <typename T>
__global__ void __launch_bounds__(ILU0_SCAN_TILE) ilu0_scan_tiles(Ilu0Params<T> p) {
    __shared__ int s_w[32];
    const int64_t i = (int64_t)blockIdx.x * ILU0_SCAN_TILE + threadIdx.x;
    const int v = i < p.n ? p.cnt[i] : 0;
    const int incl = block_inclusive_scan_1024(v, s_w);
    if (threadIdx.x == ILU0_SCAN_TILE - 1) p.tile_sum[blockIdx.x] = incl;
}

template <typename T>
__global__ void __launch_bounds__(ILU0_SCAN_TILE) ilu0_scan_sums(Ilu0Params<T> p, int ntiles) {
    __shared__ int s_w[32];
    int carry = 0;
    for (int t0 = 0; t0 < ntiles; t0 += ILU0_SCAN_TILE) {
        const int t = t0 + (int)threadIdx.x;
        const int v = t < ntiles ? p.tile_sum[t] : 0;
        const int incl = block_inclusive_scan_1024(v, s_w);
        if (t < ntiles) p.tile_sum[t] = carry + incl - v;   // exclusive offset of tile t
        carry += s_w[31];
    }
    if (threadIdx.x == 0) p.dep_ptr[p.n] = carry;
}

template <typename T>
__global__ void __launch_bounds__(ILU0_SCAN_TILE) ilu0_scan_apply(Ilu0Params<T> p) {
    __shared__ int s_w[32];
    const int64_t i = (int64_t)blockIdx.x * ILU0_SCAN_TILE + threadIdx.x;
    const int v = i < p.n ? p.cnt[i] : 0;
    const int incl = block_inclusive_scan_1024(v, s_w);
    if (i < p.n) {
        p.dep_ptr[i] = p.tile_sum[blockIdx.x] + incl - v;
        p.cnt[i] = 0;
    }
}

// 3. dependent lists (the order within a list only decides queue order)
template <typename T>
__global__ void __launch_bounds__(256) ilu0_fill(Ilu0Params<T> p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    for (int q = p.rp[i]; q < p.rp[i + 1]; ++q) {
        const int k = p.ci[q];
        if (k >= i) break;
        p.dep_idx[p.dep_ptr[k] + atomicAdd(p.cnt + k, 1)] = i;
    }
}

// 3b. per-row structure records: everything static that the factorisation
//     of a row reads before its pivot values (extents, columns, pivot
//     positions, dependents) in one 256-byte record, so that it arrives in
//     one round trip and can be fetched ahead for the rows a row readies.
//     Rows of more than 16 entries or 14 dependents get no record (-1).
//     The row's published values are set to the sentinel here.
template <typename T>
__global__ void __launch_bounds__(256) ilu0_records(Ilu0Params<T> p) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t i64 = t / ILU0_REC_LANES;
    if (i64 >= p.n) return;
    const int i = (int)i64, q = (int)(t % ILU0_REC_LANES);
    const int s = p.rp[i], e = p.rp[i + 1];
    const int d0 = p.dep_ptr[i], d1 = p.dep_ptr[i + 1];
    const int len = e - s, nd = d1 - d0;
    const bool big = len > ILU0_REC_LANES || nd > ILU0_REC_LANES - 2;
    int4 r = make_int4(INT_MAX, -1, 0, -1);
    if (!big && q < len) {
        r.x = p.ci[s + q];
        if (r.x < i) {
            const int2 pv = p.piv[s + q];
            r.y = pv.x;
            r.z = pv.y;
        }
    }
    if (!big && q < nd) r.w = p.dep_idx[d0 + q];
    if (q == ILU0_REC_LANES - 2) r.w = s;
    if (q == ILU0_REC_LANES - 1) r.w = big ? -1 : (len | (nd << 8));
    p.rec[i64 * ILU0_REC_LANES + q] = r;
    // the row's published values start as the sentinel (16 lanes per row,
    // consecutive entries)
    for (int u = s + q; u < e; u += ILU0_REC_LANES) set_sentinel(p.pub + u);
}

__device__ __forceinline__ void stop(int* abort, int* status, int bit) {
    atomicOr(status, bit);
    atomicExch(abort, 1);
}

// Pivot row k's published value at position q, polled while it is still
// the sentinel; after every 64 polls the row's done flag is acquired (set
// when a value the row published is the sentinel's bit pattern itself: the
// value read after it is then final) and the abort word read.  False in
// `fail` only when the wait ends without the value.
template <typename T>
__device__ T pub_wait(const Ilu0Params<T>& p, int64_t q, int k, bool& fail) {
    for (int it = 0;; ++it) {
        const T x = ld_relaxed(p.pub + q);
        if (!is_sentinel(x)) return x;
        if ((it & 63) == 63) {
            if (ld_acquire(p.done + k)) return ld_relaxed(p.pub + q);
            if (ld_relaxed(p.abort)) {
                fail = true;
                return T(0);
            }
        }
        if (it >= ILU0_SPIN_LIMIT) {
            stop(p.abort, p.status, ILU0_WAIT_TIMEOUT);
            fail = true;
            return T(0);
        }
        __nanosleep(32);
    }
}

// Row k's level (optional output), polled while it is still -1.
template <typename T>
__device__ int depth_wait(const Ilu0Params<T>& p, int k, bool& fail) {
    for (int it = 0;; ++it) {
        const int x = ld_relaxed(p.depth + k);
        if (x >= 0) return x;
        if (it >= ILU0_SPIN_LIMIT) {
            stop(p.abort, p.status, ILU0_WAIT_TIMEOUT);
            fail = true;
            return 0;
        }
        __nanosleep(32);
    }
}

// Row i in global memory (any length): the page's steps, lanes sharing the
// updates of each elimination step.
template <typename T>
__device__ bool factor_row_long(const Ilu0Params<T>& p, int i, int s, int e, int lane,
                                int& dmax) {
    for (int nz = s; nz < e; ++nz) {
        const int k = p.ci[nz];
        if (k >= i) break;                  // past the lower triangle (columns ascend)
        // the pivot a_kk: the first position of column k in row k
        const int ks = p.rp[k], ke = p.rp[k + 1];
        int dp = -1;
        for (int q0 = ks; q0 < ke && dp < 0; q0 += 32) {
            const unsigned hit = __ballot_sync(FULL, q0 + lane < ke && p.ci[q0 + lane] == k);
            if (hit) dp = q0 + __ffs(hit) - 1;
        }
        bool fail = false;
        const T akk = dp >= 0 ? pub_wait<T>(p, dp, k, fail) : T(0);   // warp-uniform
        if (__any_sync(FULL, fail)) return false;
        if (dp < 0 || akk == T(0)) {
            if (lane == 0) stop(p.abort, p.status, ILU0_SINGULAR);
            return false;
        }
        // every lane reads a_ik; lane 0 stores the ratio over it only after the
        // updates below, behind a warp barrier, so that no lane that runs late
        // can read the ratio in place of a_ik
        const T ratio = div_rn(__ldcg(p.v + nz), akk);
        // a_ij -= ratio * a_kj for the columns j > k of row k stored in row i
        bool bad = false;
        for (int knz = dp + 1 + lane; knz < ke; knz += 32) {
            const int j = p.ci[knz];
            int ij = -1;
            for (int q = s; q < e; ++q)
                if (p.ci[q] == j) {
                    ij = q;
                    break;
                }
            if (ij >= 0) {
                const T akj = pub_wait<T>(p, knz, k, bad);
                p.v[ij] = sub_rn(__ldcg(p.v + ij), mul_rn(ratio, akj));
            }
        }
        __syncwarp();
        if (lane == 0) p.v[nz] = ratio;
        __syncwarp();                       // the updates before the next step reads them
        if (__any_sync(FULL, bad)) return false;
        if (p.depth) dmax = max(dmax, depth_wait<T>(p, k, bad));
        if (__any_sync(FULL, bad)) return false;
    }
    return true;
}

// Row i of at most 32 entries, held in registers (lane q: entry q, loaded by
// the caller with the entry's pivot record) from the first load to the final
// store.  The pivot rows (from each pivot on) are read all at once when they
// hold at most 32 entries together, else 32 entries at a time.  Same steps
// and operations as the page, so the same bits.
template <typename T>
__device__ bool factor_row_short(const Ilu0Params<T>& p, int i, int s, int e, int lane,
                                 int my_c, T& my_v, int2 my_piv, int& dmax) {
    const int li = e - s;
    const bool mine = lane < li;
    const int nlower = __popc(__ballot_sync(FULL, mine && my_c < i));   // columns ascend
    // the pivot rows from their pivots on: row k_t is entries [dp_t, ke_t)
    const bool has = lane < nlower;
    const int len = has ? (my_piv.x >= 0 ? my_piv.y - my_piv.x : 0) : 0;
    int incl = len;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(FULL, incl, off);
        if (lane >= off) incl += y;
    }
    const int total = __shfl_sync(FULL, incl, 31);
    const int off_me = incl - len;                  // lane t: where row k_t starts in the batch
    // batch all pivot rows into the warp's lanes when they fit (one round of loads)
    int kc = -1;
    T kv = T(0);
    const bool batched = total <= 32;               // warp-uniform
    if (batched) {
        // lane L < total takes entry L - off_t of row k_t, t the last non-empty
        // row with off_t <= L (offsets ascend with t)
        int base = 0, krow = 0;
        for (int t = 0; t < nlower; ++t) {
            const int o = __shfl_sync(FULL, off_me, t);
            const int ln = __shfl_sync(FULL, len, t);
            const int dp = __shfl_sync(FULL, my_piv.x, t);
            const int col = __shfl_sync(FULL, my_c, t);
            if (ln > 0 && lane >= o) {
                base = dp - o;
                krow = col;
            }
        }
        bool fail = false;
        if (lane < total) {
            kc = p.ci[base + lane];
            kv = pub_wait<T>(p, base + lane, krow, fail);
        }
        if (__any_sync(FULL, fail)) return false;
    }
    for (int t = 0; t < nlower; ++t) {
        const int dp = __shfl_sync(FULL, my_piv.x, t);
        const int ke = __shfl_sync(FULL, my_piv.y, t);
        if (dp < 0) {                               // row k stores no pivot
            if (lane == 0) stop(p.abort, p.status, ILU0_SINGULAR);
            return false;
        }
        const T aik = __shfl_sync(FULL, my_v, t);
        if (batched) {
            const int o = __shfl_sync(FULL, off_me, t);
            const int ln = ke - dp;
            const T akk = __shfl_sync(FULL, kv, o);
            if (akk == T(0)) {
                if (lane == 0) stop(p.abort, p.status, ILU0_SINGULAR);
                return false;
            }
            const T ratio = div_rn(aik, akk);
            if (lane == t) my_v = ratio;
            // a_ij -= ratio * a_kj for the entries j > k of row k that row i stores
            for (int q = 1; q < ln; ++q) {
                const int j = __shfl_sync(FULL, kc, o + q);
                const T akj = __shfl_sync(FULL, kv, o + q);
                if (mine && my_c == j) my_v = sub_rn(my_v, mul_rn(ratio, akj));
            }
        } else {
            T ratio = T(0);
            for (int q0 = dp; q0 < ke; q0 += 32) {
                const bool have = q0 + lane < ke;
                const int c = have ? p.ci[q0 + lane] : -1;
                bool fail = false;
                const int krow = __shfl_sync(FULL, my_c, t);
                const T v = have ? pub_wait<T>(p, q0 + lane, krow, fail) : T(0);
                if (__any_sync(FULL, fail)) return false;
                int first = 0;
                if (q0 == dp) {
                    const T akk = __shfl_sync(FULL, v, 0);
                    if (akk == T(0)) {
                        if (lane == 0) stop(p.abort, p.status, ILU0_SINGULAR);
                        return false;
                    }
                    ratio = div_rn(aik, akk);
                    if (lane == t) my_v = ratio;
                    first = 1;
                }
                const int cnt = min(32, ke - q0);
                for (int q = first; q < cnt; ++q) {
                    const int j = __shfl_sync(FULL, c, q);
                    const T akj = __shfl_sync(FULL, v, q);
                    if (mine && my_c == j) my_v = sub_rn(my_v, mul_rn(ratio, akj));
                }
            }
        }
    }
    if (p.depth) {
        bool bad = false;
        int d = lane < nlower ? depth_wait<T>(p, my_c, bad) : -1;
        if (__any_sync(FULL, bad)) return false;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) d = max(d, __shfl_xor_sync(FULL, d, off));
        dmax = d;
    }
    if (mine) {
        p.v[s + lane] = my_v;
        st_relaxed(p.pub + s + lane, my_v);
    }
    return true;
}

// 4. the factorisation, one warp per ready row.  A warp that makes rows ready
// by finishing its own keeps the first of them (no queue round trip on the
// critical path) and queues the rest.  Waiting warps give up only when no
// row has finished anywhere for ILU0_SPIN_LIMIT polls, or on the abort word.
//
// A row's structure, its own values (no other row writes them) and its
// dependents need no ordering; its pivot rows' values are their published
// values, waited for while they are still the sentinel.  No fence and no
// acquire-release pair lies on the path from one row to the next
// (measured on GB300, the 707 x 707 Laplacian in binary64: 5.07 ms per call
// against 5.76 ms with acquire-release count-downs and the values read after
// the acquire; bit for bit the same factors).
template <typename T>
__global__ void __launch_bounds__(ILU0_THREADS, 2) ilu0_factor(Ilu0Params<T> p) {
    const int lane = threadIdx.x & 31;
    const int4 NOREC = make_int4(INT_MAX, -1, 0, -1);
    int next = -1;                              // a row this warp made ready
    int4 next_rc = NOREC;                       // its record, when fetched ahead
    bool next_has = false;
    for (;;) {
        int i = next;
        int4 rc = next_rc;
        const bool have = next_has;
        next = -1;
        next_has = false;
        const bool kept = i >= 0;
        if (!kept) {
            int h = 0;
            if (lane == 0) h = atomicAdd(p.head, 1);
            h = __shfl_sync(FULL, h, 0);
            if (h >= p.n) return;
            // wait for slot h to be filled, or for every row to be finished
            int seen = -1;
            for (int it = 0;; ++it) {
                i = ld_relaxed(p.queue + h);
                if (__all_sync(FULL, i >= 0)) break;
                // the shared words every SPMM_ILU0_POLL_EVERY polls (they are hot lines)
                if ((it & (SPMM_ILU0_POLL_EVERY - 1)) == SPMM_ILU0_POLL_EVERY - 1) {
                    int ab = 0, fin = 0;
                    if (lane == 0) {
                        ab = ld_relaxed(p.abort);
                        fin = ld_relaxed(p.finished);
                    }
                    ab = __shfl_sync(FULL, ab, 0);
                    fin = __shfl_sync(FULL, fin, 0);
                    if (ab != 0 || fin >= p.n) return;
                    if (fin != seen) {           // progress somewhere: keep waiting
                        seen = fin;
                        it = 0;
                    }
                }
                if (it >= ILU0_SPIN_LIMIT) {
                    if (lane == 0) stop(p.abort, p.status, ILU0_WAIT_TIMEOUT);
                    return;
                }
                __nanosleep(SPMM_ILU0_SLEEP_NS);
            }
        }
        // row i's structure record (already here when fetched ahead)
        if (!have) rc = lane < ILU0_REC_LANES ? p.rec[(int64_t)i * ILU0_REC_LANES + lane] : NOREC;
        const int meta = __shfl_sync(FULL, rc.w, ILU0_REC_LANES - 1);
        const int s = __shfl_sync(FULL, rc.w, ILU0_REC_LANES - 2);
        int e, d0 = 0, nd;
        bool short_row;
        int my_c = INT_MAX;
        T my_v = T(0);
        int2 my_piv = make_int2(-1, 0);
        int dj = -1;
        int dep0 = -1, dep1 = -1;
        int4 pf0 = NOREC, pf1 = NOREC;
        if (meta >= 0) {
            // from the record: at most 16 entries, at most 14 dependents
            const int len = meta & 0xff;
            nd = meta >> 8;
            e = s + len;
            short_row = true;
            my_c = rc.x;
            my_piv = make_int2(rc.y, rc.z);
            if (lane < len) my_v = __ldcg(p.v + s + lane);   // written by row i only
            dj = lane < nd ? rc.w : -1;
            // fetch the first two dependents' records ahead: one of them is
            // likely the row this one readies and keeps
            dep0 = nd > 0 ? __shfl_sync(FULL, rc.w, 0) : -1;
            dep1 = nd > 1 ? __shfl_sync(FULL, rc.w, 1) : -1;
            if (SPMM_ILU0_PREFETCH && lane < ILU0_REC_LANES) {
                if (dep0 >= 0) pf0 = p.rec[(int64_t)dep0 * ILU0_REC_LANES + lane];
                if (dep1 >= 0) pf1 = p.rec[(int64_t)dep1 * ILU0_REC_LANES + lane];
            }
        } else {
            // no record: extents, entries, pivot records and dependents from the arrays
            e = p.rp[i + 1];
            d0 = p.dep_ptr[i];
            nd = p.dep_ptr[i + 1] - d0;
            short_row = e - s <= 32;
            if (short_row && lane < e - s) {
                my_c = p.ci[s + lane];
                my_v = __ldcg(p.v + s + lane);
                if (my_c < i) my_piv = p.piv[s + lane];
            }
            dj = lane < nd ? p.dep_idx[d0 + lane] : -1;
        }
        int dmax = -1;
        bool ok;
        if (short_row)
            ok = factor_row_short<T>(p, i, s, e, lane, my_c, my_v, my_piv, dmax);
        else
            ok = factor_row_long<T>(p, i, s, e, lane, dmax);
        if (!ok) return;
        if (!short_row) {                       // publish the long row's final values
            __syncwarp();
            for (int q = s + lane; q < e; q += 32) st_relaxed(p.pub + q, __ldcg(p.v + q));
        }
        {
            // a published value equal to the sentinel: say so by the done flag
            bool sent = false;
            if (short_row) sent = lane < e - s && is_sentinel(my_v);
            else
                for (int q = s + lane; q < e; q += 32) sent |= is_sentinel(__ldcg(p.v + q));
            if (__any_sync(FULL, sent)) {
                __syncwarp();                   // every lane's stores before the release
                if (lane == 0) st_release(p.done + i, 1);
            }
        }
        if (p.depth && lane == 0) st_relaxed(p.depth + i, dmax + 1);
        // count down the rows that wait for row i (relaxed: they only schedule;
        // the values travel as published values); keep one, queue the rest
        __syncwarp();
        for (int c = 0; c < nd; c += 32) {
            const int j = c == 0 ? dj : (c + lane < nd ? p.dep_idx[d0 + c + lane] : -1);
            bool ready = false;
            if (c + lane < nd) ready = atomicAdd(p.pending + j, -1) == 1;
            unsigned rm = __ballot_sync(FULL, ready);
            if (next < 0 && rm) {
                const int keep = __ffs(rm) - 1;
                next = __shfl_sync(FULL, j, keep);
                if (lane == keep) ready = false;
                rm &= rm - 1;
                if (SPMM_ILU0_PREFETCH && next == dep0) {
                    next_rc = pf0;
                    next_has = true;
                } else if (SPMM_ILU0_PREFETCH && next == dep1) {
                    next_rc = pf1;
                    next_has = true;
                }
            }
            if (ready) st_relaxed(p.queue + atomicAdd(p.tail, 1), j);
        }
        __syncwarp();
        if (lane == 0) atomicAdd(p.finished, 1);
    }
}

}  // namespace

template <typename T>
cudaError_t launch_ilu0(const Ilu0Params<T>& p, int grid, cudaStream_t st) {
    const int rb = (p.n + 255) / 256;
    ilu0_count<T><<<rb, 256, 0, st>>>(p);
    const int ntiles = (int)(((int64_t)p.n + ILU0_SCAN_TILE - 1) / ILU0_SCAN_TILE);
    ilu0_scan_tiles<T><<<ntiles, ILU0_SCAN_TILE, 0, st>>>(p);
    ilu0_scan_sums<T><<<1, ILU0_SCAN_TILE, 0, st>>>(p, ntiles);
    ilu0_scan_apply<T><<<ntiles, ILU0_SCAN_TILE, 0, st>>>(p);
    ilu0_fill<T><<<rb, 256, 0, st>>>(p);
    ilu0_records<T><<<(unsigned)(((int64_t)p.n * ILU0_REC_LANES + 255) / 256), 256, 0, st>>>(p);
    ilu0_factor<T><<<grid, ILU0_THREADS, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename T>
int ilu0_blocks_per_sm() {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, ilu0_factor<T>, ILU0_THREADS, 0) !=
            cudaSuccess || b < 1) {
        cudaGetLastError();
        b = 1;
    }
    return SPMM_ILU0_BLOCKS_PER_SM > 0 ? std::min(b, SPMM_ILU0_BLOCKS_PER_SM) : b;
}

template cudaError_t launch_ilu0<float>(const Ilu0Params<float>&, int, cudaStream_t);
template cudaError_t launch_ilu0<double>(const Ilu0Params<double>&, int, cudaStream_t);
template int ilu0_blocks_per_sm<float>();
template int ilu0_blocks_per_sm<double>();

}  // namespace spmm
