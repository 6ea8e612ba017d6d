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
        // beta == +1 / -1 with 16-byte vectors and one slot per lane: the
        // epilogue leaves out the binary64 multiply by beta (exact, so the
        // same bits); this path is bound by binary64 throughput on GB300
        // (5-point Laplacian, alpha = 2, beta = -1: 0.248 -> 0.216 ms)
        if constexpr (W == 2 && R == 1) {
            if (p.beta == 1.0)
                return launch_windowed(rows_kernel<double, W, G, R, true, false, 1>, gd, bd, 0, st,
                                       overlap, win, p);
            if (p.beta == -1.0)
                return launch_windowed(rows_kernel<double, W, G, R, true, false, -1>, gd, bd, 0,
                                       st, overlap, win, p);
        }
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
