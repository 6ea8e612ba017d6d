// One-launch small-product kernel instantiations for float (m <= SMALL_ROWS).
// The instances mirror launch_rows<float>, so that short and medium rows get
// the binned path's results bit for bit.
#include "spmm_dispatch.cuh"
#include "spmm_kernels.cuh"

namespace spmm {

template <>
cudaError_t launch_small<float>(const SpmmParams<float>& p, const Geometry& g, int short_max,
                                int grid, cudaStream_t st, const L2Window* win) {
    return dispatch_geometry<float>(g, [&]<int W, int G, int R>() -> cudaError_t {
        const dim3 gd(grid), bd(RowsOccupancy<float, W, G>::THREADS);
        if constexpr (G == 32 && R == 1 && W > 1) {
            if (g.whole) {
                if (p.beta != float(0))
                    return launch_windowed(small_kernel<float, W, G, R, true, true>, gd, bd, 0, st,
                                           false, win, p, short_max);
                return launch_windowed(small_kernel<float, W, G, R, false, true>, gd, bd, 0, st,
                                       false, win, p, short_max);
            }
        }
        if (p.beta != float(0))
            return launch_windowed(small_kernel<float, W, G, R, true, false>, gd, bd, 0, st, false,
                                   win, p, short_max);
        return launch_windowed(small_kernel<float, W, G, R, false, false>, gd, bd, 0, st, false,
                               win, p, short_max);
    });
}

}  // namespace spmm
