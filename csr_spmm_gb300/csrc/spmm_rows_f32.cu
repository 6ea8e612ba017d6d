// Short/medium-row kernel instantiations for float.
#include "spmm_dispatch.cuh"
#include "spmm_kernels.cuh"

namespace spmm {

template <>
cudaError_t launch_rows<float>(const SpmmParams<float>& p, const Geometry& g, int grid,
                               cudaStream_t st, bool overlap, const L2Window* win) {
    return dispatch_geometry<float>(g, [&]<int W, int G, int R>() -> cudaError_t {
        const dim3 gd(grid), bd(RowsOccupancy<float, W, G>::THREADS);
        // whole-vector instances for full-warp lane groups: 22% fewer instructions
        // and 10% less time on GB300; for narrower groups the general code is
        // faster (it spills less), and in binary64 it is too
        if constexpr (G == 32 && R == 1 && W > 1) {
            if (g.whole) {
                if (p.beta != float(0))
                    return launch_windowed(rows_kernel<float, W, G, R, true, true>, gd, bd, 0, st,
                                           overlap, win, p);
                return launch_windowed(rows_kernel<float, W, G, R, false, true>, gd, bd, 0, st,
                                       overlap, win, p);
            }
        }
        if (p.beta != float(0))
            return launch_windowed(rows_kernel<float, W, G, R, true, false>, gd, bd, 0, st, overlap,
                                   win, p);
        return launch_windowed(rows_kernel<float, W, G, R, false, false>, gd, bd, 0, st, overlap, win,
                               p);
    });
}

template <>
int rows_blocks_per_sm<float>(const Geometry& g) {
    int blocks = 0;
    cudaError_t e = dispatch_geometry<float>(g, [&]<int W, int G, int R>() -> cudaError_t {
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &blocks, rows_kernel<float, W, G, R, false, false>, RowsOccupancy<float, W, G>::THREADS,
            0);
    });
    return (e == cudaSuccess && blocks > 0) ? blocks : 1;
}

}  // namespace spmm
