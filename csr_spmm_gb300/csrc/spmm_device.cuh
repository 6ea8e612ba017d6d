// Device-side building blocks shared by the CSR SpMM kernels (sm_103a).
//
// Loads carry explicit cache policy:
//   * B rows are gathered through the non-coherent path with default
//     allocation (see BLoad);
//   * the CSR stream (col_idx, values) is read once, with L1::no_allocate and
//     an L2 evict_first policy, so it does not displace B;
//   * C is read (beta != 0) and written with the streaming (.cs) policy.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "spmm_internal.h"

namespace spmm {

// ---------------------------------------------------------------------------
// cache policies (created once per thread; cheap)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------------------
// CSR stream loads (read once)
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ld_stream(const int* p, uint64_t pol) {
    int v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.b32 %0, [%1], %2;"
                 : "=r"(v) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ float ld_stream(const float* p, uint64_t pol) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.f32 %0, [%1], %2;"
                 : "=f"(v) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ double ld_stream(const double* p, uint64_t pol) {
    double v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.f64 %0, [%1], %2;"
                 : "=d"(v) : "l"(p), "l"(pol));
    return v;
}

// ---------------------------------------------------------------------------
// B gathers: W consecutive elements (W * sizeof(T) = 4, 8 or 16 bytes) through
// the non-coherent path with default L1/L2 allocation.  Measured on GB300 for
// random row gathers, this beats both an L2 evict_last policy and
// L1::no_allocate at every span tried (32 MB .. 2 GB).
// ---------------------------------------------------------------------------
template <typename T, int W> struct BLoad;

template <> struct BLoad<float, 1> {
    __device__ __forceinline__ static void run(const float* p, float (&v)[1]) {
        asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v[0]) : "l"(p));
    }
};
template <> struct BLoad<float, 4> {
    __device__ __forceinline__ static void run(const float* p, float (&v)[4]) {
        asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "l"(p));
    }
};
template <> struct BLoad<double, 1> {
    __device__ __forceinline__ static void run(const double* p, double (&v)[1]) {
        asm volatile("ld.global.nc.f64 %0, [%1];" : "=d"(v[0]) : "l"(p));
    }
};
template <> struct BLoad<double, 2> {
    __device__ __forceinline__ static void run(const double* p, double (&v)[2]) {
        asm volatile("ld.global.nc.v2.f64 {%0,%1}, [%2];" : "=d"(v[0]), "=d"(v[1]) : "l"(p));
    }
};

// Element-wise load of the first `cnt` (< W) elements; the rest are zero.
template <typename T, int W>
__device__ __forceinline__ void load_b_partial(const T* p, int cnt, T (&v)[W]) {
#pragma unroll
    for (int e = 0; e < W; ++e) {
        T x[1] = {T(0)};
        if (e < cnt) BLoad<T, 1>::run(p + e, x);
        v[e] = x[0];
    }
}

// ---------------------------------------------------------------------------
// C epilogue: C = alpha * acc (beta == 0, C not read) or alpha * acc + beta * C,
// evaluated as fma(alpha, acc, beta * C).  BS = +1 / -1 marks a kernel built
// for beta == +1 / -1: beta * C is then +C / -C exactly, so the multiply is
// left out and the result is bit for bit that of the general form.  (On GB300
// binary64 arithmetic is scarce, and the multiply is a quarter of the FP64
// work of a 5-point-stencil product.)
// ---------------------------------------------------------------------------
template <typename T, int BS = 0>
__device__ __forceinline__ T epi(T alpha, T acc, T beta, T c_old) {
    static_assert(BS == 0 || BS == 1 || BS == -1, "beta sign: 0 (any beta), +1 or -1");
    if constexpr (BS == 1) return fma(alpha, acc, c_old);
    else if constexpr (BS == -1) return fma(alpha, acc, -c_old);
    else return fma(alpha, acc, beta * c_old);
}

// Output store: streaming (.cs) by default; `keep` stores with the default
// policy instead, for an output that the next product of a chain reads back.
template <typename V>
__device__ __forceinline__ void st_out(V* q, V o, bool keep) {
    if (keep) *q = o;
    else __stcs(q, o);
}

template <typename T, int W>
__device__ __forceinline__ void store_c(T* c, int cnt, const T (&acc)[W], T alpha, T beta,
                                        bool read_c, bool keep = false) {
    if (cnt == W && (W * sizeof(T)) % 16 == 0) {
        // W * sizeof(T) is 16 or 32 bytes: use 16-byte streaming accesses
        constexpr int PER = 16 / sizeof(T);
#pragma unroll
        for (int h = 0; h < W; h += PER) {
            if constexpr (sizeof(T) == 4) {
                float4* q = reinterpret_cast<float4*>(c + h);
                float4 o;
                if (read_c) {
                    float4 old = __ldcs(q);
                    o = make_float4(epi<float>(alpha, acc[h], beta, old.x),
                                    epi<float>(alpha, acc[h + 1], beta, old.y),
                                    epi<float>(alpha, acc[h + 2], beta, old.z),
                                    epi<float>(alpha, acc[h + 3], beta, old.w));
                } else {
                    o = make_float4(alpha * acc[h], alpha * acc[h + 1], alpha * acc[h + 2],
                                    alpha * acc[h + 3]);
                }
                st_out(q, o, keep);
            } else {
                double2* q = reinterpret_cast<double2*>(c + h);
                double2 o;
                if (read_c) {
                    double2 old = __ldcs(q);
                    o = make_double2(epi<double>(alpha, acc[h], beta, old.x),
                                     epi<double>(alpha, acc[h + 1], beta, old.y));
                } else {
                    o = make_double2(alpha * acc[h], alpha * acc[h + 1]);
                }
                st_out(q, o, keep);
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < W; ++e) {
            if (e < cnt) {
                T o = read_c ? epi<T>(alpha, acc[e], beta, __ldcs(c + e)) : alpha * acc[e];
                st_out(c + e, o, keep);
            }
        }
    }
}

// C elements [0, cnt) of a vector slot, streaming load (the rest stay zero).
template <typename T, int W>
__device__ __forceinline__ void load_c(const T* c, int cnt, T (&v)[W]) {
    if (cnt == W && (W * sizeof(T)) % 16 == 0) {
        constexpr int PER = 16 / sizeof(T);
#pragma unroll
        for (int h = 0; h < W; h += PER) {
            if constexpr (sizeof(T) == 4) {
                const float4 x = __ldcs(reinterpret_cast<const float4*>(c + h));
                v[h] = x.x; v[h + 1] = x.y; v[h + 2] = x.z; v[h + 3] = x.w;
            } else {
                const double2 x = __ldcs(reinterpret_cast<const double2*>(c + h));
                v[h] = x.x; v[h + 1] = x.y;
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < W; ++e)
            if (e < cnt) v[e] = __ldcs(c + e);
    }
}

// C = alpha * acc + beta * c0 with c0 already loaded (BS: see epi).
template <typename T, int W, int BS = 0>
__device__ __forceinline__ void store_c_pre(T* c, int cnt, const T (&acc)[W], const T (&c0)[W],
                                            T alpha, T beta) {
    T o[W];
#pragma unroll
    for (int e = 0; e < W; ++e) o[e] = epi<T, BS>(alpha, acc[e], beta, c0[e]);
    if (cnt == W && (W * sizeof(T)) % 16 == 0) {
        constexpr int PER = 16 / sizeof(T);
#pragma unroll
        for (int h = 0; h < W; h += PER) {
            if constexpr (sizeof(T) == 4)
                __stcs(reinterpret_cast<float4*>(c + h), make_float4(o[h], o[h + 1], o[h + 2], o[h + 3]));
            else
                __stcs(reinterpret_cast<double2*>(c + h), make_double2(o[h], o[h + 1]));
        }
    } else {
#pragma unroll
        for (int e = 0; e < W; ++e)
            if (e < cnt) __stcs(c + e, o[e]);
    }
}

}  // namespace spmm
