// Maps a run-time Geometry onto the compiled (W, G, R) instantiations.
#pragma once

#include "spmm_internal.h"

namespace spmm {

// f is a generic lambda  [&]<int W, int G, int R>() -> cudaError_t
template <typename T, int W, typename F>
cudaError_t dispatch_gr(const Geometry& g, F& f) {
    if (g.R == 1) {
        switch (g.G) {
            case 1: return f.template operator()<W, 1, 1>();
            case 2: return f.template operator()<W, 2, 1>();
            case 4: return f.template operator()<W, 4, 1>();
            case 8: return f.template operator()<W, 8, 1>();
            case 16: return f.template operator()<W, 16, 1>();
            case 32: return f.template operator()<W, 32, 1>();
            default: return cudaErrorInvalidValue;
        }
    }
    if (g.G == 32 && g.R == 2) return f.template operator()<W, 32, 2>();
    if (g.G == 32 && g.R == 4) return f.template operator()<W, 32, 4>();
    return cudaErrorInvalidValue;
}

template <typename T, typename F>
cudaError_t dispatch_geometry(const Geometry& g, F&& f) {
    constexpr int WV = 16 / (int)sizeof(T);    // one 16-byte vector
    if (g.W == WV) return dispatch_gr<T, WV>(g, f);
    if (g.W == 1) return dispatch_gr<T, 1>(g, f);
    return cudaErrorInvalidValue;
}

}  // namespace spmm
