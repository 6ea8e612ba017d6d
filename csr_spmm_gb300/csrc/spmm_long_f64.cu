// Long-row CTA-split (with its in-launch fixup) instantiations for double.
#include "spmm_dispatch.cuh"
#include "spmm_kernels.cuh"

namespace spmm {

template <>
cudaError_t launch_long<double>(const SpmmParams<double>& p, const Geometry& g, cudaStream_t st,
                            bool overlap, const L2Window* win) {
    return dispatch_geometry<double>(g, [&]<int W, int G, int R>() -> cudaError_t {
        const size_t smem = (size_t)LONG_WARPS * G * R * W * sizeof(double);
        auto kern = long_kernel<double, W, G, R>;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
        }
        return launch_windowed(kern, dim3(p.long_grid), dim3(LONG_THREADS), smem, st, overlap, win, p);
    });
}

}  // namespace spmm
