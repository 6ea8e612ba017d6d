// Short/medium-row kernel instantiations for double.
#include "spmm_dispatch.cuh"
#include "spmm_kernels.cuh"

namespace spmm {

template <>
cudaError_t launch_rows<double>(const SpmmParams<double>& p, const Geometry& g, int grid,
                               cudaStream_t st, bool overlap, const L2Window* win) {
    return dispatch_geometry<double>(g, [&]<int W, int G, int R>() -> cudaError_t {
        const dim3 gd(grid), bd(RowsOccupancy<double, W, G>::THREADS);
        // (whole-vector instances are binary32 only: measured slower in binary64)
        if (p.beta != double(0))
            return launch_windowed(rows_kernel<double, W, G, R, true, false>, gd, bd, 0, st, overlap,
                                   win, p);
        return launch_windowed(rows_kernel<double, W, G, R, false, false>, gd, bd, 0, st, overlap, win,
                               p);
    });
}

template <>
int rows_blocks_per_sm<double>(const Geometry& g) {
    int blocks = 0;
    cudaError_t e = dispatch_geometry<double>(g, [&]<int W, int G, int R>() -> cudaError_t {
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &blocks, rows_kernel<double, W, G, R, false, false>, RowsOccupancy<double, W, G>::THREADS,
            0);
    });
    return (e == cudaSuccess && blocks > 0) ? blocks : 1;
}

}  // namespace spmm
