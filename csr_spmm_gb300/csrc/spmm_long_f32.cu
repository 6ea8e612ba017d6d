// Long-row CTA-split (with its in-launch fixup) instantiations for float.
#include "spmm_dispatch.cuh"
#include "spmm_kernels.cuh"

namespace spmm {

template <>
cudaError_t launch_long<float>(const SpmmParams<float>& p, const Geometry& g, cudaStream_t st,
                            bool overlap, const L2Window* win) {
    return dispatch_geometry<float>(g, [&]<int W, int G, int R>() -> cudaError_t {
        const size_t smem = (size_t)LONG_WARPS * G * R * W * sizeof(float);
        auto kern = long_kernel<float, W, G, R>;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
        }
        return launch_windowed(kern, dim3(p.long_grid), dim3(LONG_THREADS), smem, st, overlap, win, p);
    });
}

}  // namespace spmm
