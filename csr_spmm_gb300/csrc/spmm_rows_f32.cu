// Short/medium-row kernel instantiations for float.
#include "spmm_dispatch.cuh"
#include "spmm_kernels.cuh"

namespace spmm {

template <>
cudaError_t launch_rows<float>(const SpmmParams<float>& p, const Geometry& g, int grid,
                               cudaStream_t st, bool overlap, const L2Window* win) {
    return dispatch_geometry<float>(g, [&]<int W, int G, int R>() -> cudaError_t {
        if (p.beta != float(0))
            return launch_windowed(rows_kernel<float, W, G, R, true>, dim3(grid), dim3(ROWS_THREADS),
                                  0, st, overlap, win, p);
        return launch_windowed(rows_kernel<float, W, G, R, false>, dim3(grid), dim3(ROWS_THREADS), 0,
                              st, overlap, win, p);
    });
}

template <>
int rows_blocks_per_sm<float>(const Geometry& g) {
    int blocks = 0;
    cudaError_t e = dispatch_geometry<float>(g, [&]<int W, int G, int R>() -> cudaError_t {
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &blocks, rows_kernel<float, W, G, R, false>, ROWS_THREADS, 0);
    });
    return (e == cudaSuccess && blocks > 0) ? blocks : 1;
}

}  // namespace spmm
