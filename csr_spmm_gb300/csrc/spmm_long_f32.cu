// Long-row CTA-split and fixup instantiations for float.
#include "spmm_dispatch.cuh"
#include "spmm_kernels.cuh"

namespace spmm {

template <>
cudaError_t launch_long<float>(const SpmmParams<float>& p, const Geometry& g, cudaStream_t st) {
    return dispatch_geometry<float>(g, [&]<int W, int G, int R>() -> cudaError_t {
        const size_t smem = (size_t)LONG_WARPS * G * R * W * sizeof(float);
        auto kern = long_kernel<float, W, G, R>;
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
cudaError_t launch_fixup<float>(const SpmmParams<float>& p, cudaStream_t st) {
    fixup_kernel<float><<<p.long_grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace spmm
