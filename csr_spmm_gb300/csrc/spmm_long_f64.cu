// Long-row CTA-split and fixup instantiations for double.
#include "spmm_dispatch.cuh"
#include "spmm_kernels.cuh"

namespace spmm {

template <>
cudaError_t launch_long<double>(const SpmmParams<double>& p, const Geometry& g, cudaStream_t st) {
    return dispatch_geometry<double>(g, [&]<int W, int G, int R>() -> cudaError_t {
        const size_t smem = (size_t)LONG_WARPS * G * R * W * sizeof(double);
        auto kern = long_kernel<double, W, G, R>;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
        }
        kern<<<p.long_grid, LONG_THREADS, smem, st>>>(p);
        return cudaGetLastError();
    });
}

template <>
cudaError_t launch_fixup<double>(const SpmmParams<double>& p, cudaStream_t st) {
    fixup_kernel<double><<<p.long_grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace spmm
