// One-launch small-product kernel instantiations for double (m <= SMALL_ROWS).
// The instances mirror launch_rows<double> (beta = +1 / -1 epilogues
// included), so that short and medium rows get the binned path's results
// bit for bit.
#include "spmm_dispatch.cuh"
#include "spmm_kernels.cuh"

namespace spmm {

template <>
cudaError_t launch_small<double>(const SpmmParams<double>& p, const Geometry& g, int short_max,
                                 int grid, cudaStream_t st, const L2Window* win) {
    return dispatch_geometry<double>(g, [&]<int W, int G, int R>() -> cudaError_t {
        const dim3 gd(grid), bd(RowsOccupancy<double, W, G>::THREADS);
        if constexpr (W == 2 && R == 1) {
            if (p.beta == 1.0)
                return launch_windowed(small_kernel<double, W, G, R, true, false, 1>, gd, bd, 0, st,
                                       false, win, p, short_max);
            if (p.beta == -1.0)
                return launch_windowed(small_kernel<double, W, G, R, true, false, -1>, gd, bd, 0,
                                       st, false, win, p, short_max);
        }
        if (p.beta != double(0))
            return launch_windowed(small_kernel<double, W, G, R, true, false>, gd, bd, 0, st, false,
                                   win, p, short_max);
        return launch_windowed(small_kernel<double, W, G, R, false, false>, gd, bd, 0, st, false,
                               win, p, short_max);
    });
}

}  // namespace spmm
