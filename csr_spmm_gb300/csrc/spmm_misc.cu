// Epilogue-only kernel (alpha == 0 or k == 0: C = beta * C, C write-only when
// beta == 0), the CSR structure check, and the binary64 FMA throughput probe
// that the measurement of binary64 products is set against.
#include "spmm_internal.h"

namespace spmm {
namespace {

template <typename T>
__global__ void __launch_bounds__(256)
scale_kernel(T* __restrict__ C, int64_t ldc, int m, int n, T beta) {
    const int64_t total = (int64_t)m * n;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const bool read_c = beta != T(0);
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += stride) {
        const int64_t i = t / n, c = t - i * n;
        T* q = C + i * ldc + c;
        *q = read_c ? beta * *q : T(0);
    }
}

// status bits: 1 row_ptr[0] != 0, 2 row_ptr decreases, 4 row_ptr[m] != nnz,
// 8 a column index outside [0, k)
__global__ void __launch_bounds__(256)
csr_check_kernel(const int* __restrict__ row_ptr, const int* __restrict__ col_idx, int64_t m,
                 int64_t k, int64_t nnz, int* __restrict__ status) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int bits = 0;
    if (t0 == 0) {
        if (row_ptr[0] != 0) bits |= 1;
        if ((int64_t)row_ptr[m] != nnz) bits |= 4;
    }
    for (int64_t i = t0; i < m; i += stride)
        if (row_ptr[i + 1] < row_ptr[i]) bits |= 2;
    for (int64_t q = t0; q < nnz; q += stride) {
        const int c = col_idx[q];
        if (c < 0 || (int64_t)c >= k) bits |= 8;
    }
    if (bits) atomicOr(status, bits);
}

// Binary64 FMA throughput: each thread runs FMA_CHAINS independent chains of
// dependent fma.rn.f64 (a = a * x + y, x and y known only at run time) for
// `iters` steps; the chains' sum is stored so that no work is dead.
constexpr int FMA_CHAINS = 8;
__global__ void __launch_bounds__(256) fp64_fma_probe(double x, double y, int iters,
                                                      double* __restrict__ sink) {
    double a[FMA_CHAINS];
#pragma unroll
    for (int j = 0; j < FMA_CHAINS; ++j) a[j] = 1e-9 * threadIdx.x + j;
#pragma unroll 4
    for (int it = 0; it < iters; ++it)
#pragma unroll
        for (int j = 0; j < FMA_CHAINS; ++j) a[j] = fma(a[j], x, y);
    double sum = 0.0;
#pragma unroll
    for (int j = 0; j < FMA_CHAINS; ++j) sum += a[j];
    sink[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = sum;
}

}  // namespace

cudaError_t launch_fp64_fma_probe(int grid, int iters, double* sink, cudaStream_t st,
                                  int64_t* fmas) {
    fp64_fma_probe<<<grid, 256, 0, st>>>(0.999999999, 1e-12, iters, sink);
    *fmas = (int64_t)grid * 256 * FMA_CHAINS * iters;
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_scale(T* C, int64_t ldc, int m, int n, T beta, int grid, cudaStream_t st) {
    scale_kernel<T><<<grid, 256, 0, st>>>(C, ldc, m, n, beta);
    return cudaGetLastError();
}
template cudaError_t launch_scale<float>(float*, int64_t, int, int, float, int, cudaStream_t);
template cudaError_t launch_scale<double>(double*, int64_t, int, int, double, int, cudaStream_t);

cudaError_t launch_csr_check(const int* row_ptr, const int* col_idx, int64_t m, int64_t k,
                             int64_t nnz, int* status, cudaStream_t st) {
    const int64_t work = m > nnz ? m : nnz;
    int grid = (int)((work + 255) / 256);
    if (grid < 1) grid = 1;
    if (grid > 4096) grid = 4096;
    csr_check_kernel<<<grid, 256, 0, st>>>(row_ptr, col_idx, m, k, nnz, status);
    return cudaGetLastError();
}

}  // namespace spmm
