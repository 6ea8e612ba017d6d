// spmm_csr_f32_noalloc: the binary32 product for callers that must not
// allocate device memory -- code running where cudaMalloc is unavailable or
// forbidden (inside a memory-capped or pre-sized allocator, a plugin that owns
// no memory budget, a real-time loop that may not stall on allocation).  It runs
// the same kernels as spmm_csr_f32, but every byte of scratch (row bins, the
// long-row prefix and partial sums) comes from one file-scope device array of
// fixed size, so the call itself allocates nothing and needs no handle.
//
// The array is a single buffer per device, shared by every call: calls that
// overlap on the GPU (two streams, or a second call before the first has run)
// race on it.  Nothing in it has to start at zero: each call's pre-pass writes
// every word a later kernel of the same call reads (it also zeroes the
// long-row counters before the long-row kernel counts on them).
#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>

#include "csr_spmm.h"
#include "spmm_internal.h"

using namespace spmm;

namespace {

// Limits of the static scratch (see include/csr_spmm.h).
constexpr int64_t NOALLOC_MAX_ROWS = 1 << 19;      // m <= 524,288
constexpr int64_t NOALLOC_MAX_COLS = 512;          // n <= 512
constexpr int NOALLOC_LONG_GRID_MAX = 640;         // the long-row grid of up to 160 SMs

constexpr size_t al256(size_t x) { return (x + 255) / 256 * 256; }
constexpr int64_t NOALLOC_TILES = (NOALLOC_MAX_ROWS + BIN_TILE - 1) / BIN_TILE;
constexpr size_t OFF_HDR = 0;
constexpr size_t OFF_TILE_COUNTS = al256(OFF_HDR + sizeof(int) * HDR_WORDS);
constexpr size_t OFF_TILE_OFFSETS = al256(OFF_TILE_COUNTS + sizeof(int) * BIN_REC * NOALLOC_TILES);
constexpr size_t OFF_ROWLIST = al256(OFF_TILE_OFFSETS + sizeof(int) * BIN_REC * NOALLOC_TILES);
constexpr size_t OFF_MED_PRE = al256(OFF_ROWLIST + sizeof(int) * NOALLOC_MAX_ROWS);
constexpr size_t OFF_LONG_PRE = al256(OFF_MED_PRE + sizeof(int) * (NOALLOC_MAX_ROWS + 1));
constexpr size_t OFF_LONG_CNT = al256(OFF_LONG_PRE + sizeof(int) * (NOALLOC_MAX_ROWS + 1));
constexpr size_t OFF_PARTIALS = al256(OFF_LONG_CNT + sizeof(int) * NOALLOC_MAX_ROWS);
constexpr size_t NOALLOC_BYTES =
    al256(OFF_PARTIALS + sizeof(float) * 2 * NOALLOC_LONG_GRID_MAX * NOALLOC_MAX_COLS);

// The scratch itself (about 11.1 MB on every device that loads this library).
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

// Per-device set-up, done once on the first call made with that device current.
struct DeviceSetup {
    bool ready = false;
    bool supported = false;
    unsigned char* scratch = nullptr;    // device address of g_noalloc_scratch
    int num_sms = 0;
    int64_t l2_bytes = 0;
    // rows-kernel blocks per SM by geometry (an occupancy query, made once)
    struct Occ { int W, G, R, blocks; };
    Occ occ[16];
    int nocc = 0;
};
constexpr int MAX_DEVICES = 64;
DeviceSetup g_setup[MAX_DEVICES];
std::mutex g_setup_mutex;

spmm_status_t setup_device(int dev, DeviceSetup** out) {
    if (dev < 0 || dev >= MAX_DEVICES) return SPMM_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup& s = g_setup[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0, l2 = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
            cudaGetLastError();
            return SPMM_ERR_CUDA;
        }
        // the static partial sums hold NOALLOC_LONG_GRID_MAX long-row CTAs, the
        // handle path's long-row grid on devices of up to 160 SMs
        s.supported = (major == 10 && minor == 3) && long_grid_for(sms) <= NOALLOC_LONG_GRID_MAX;
        if (s.supported) {
            // In host code g_noalloc_scratch names a host-side stand-in; the
            // device address is looked up here, with `dev` current.
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
                cudaGetLastError();
                return SPMM_ERR_CUDA;
            }
            s.scratch = static_cast<unsigned char*>(p);
        }
        s.num_sms = sms;
        s.l2_bytes = l2;
        s.ready = true;
    }
    if (!s.supported) return SPMM_ERR_UNSUPPORTED_DEVICE;
    *out = &s;
    return SPMM_OK;
}

inline bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

// Rows-kernel blocks per SM for geometry g on this device (cached; the
// first call with a geometry asks the occupancy calculator).
int rows_blocks(DeviceSetup* ds, const Geometry& g) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    for (int i = 0; i < ds->nocc; ++i)
        if (ds->occ[i].W == g.W && ds->occ[i].G == g.G && ds->occ[i].R == g.R)
            return ds->occ[i].blocks;
    const int b = rows_blocks_per_sm<float>(g);
    if (ds->nocc < 16) ds->occ[ds->nocc++] = {g.W, g.G, g.R, b};
    return b;
}

}  // namespace

extern "C" spmm_status_t spmm_csr_f32_noalloc(float alpha, const int32_t* row_ptr,
                                              const int32_t* col_idx, const float* values,
                                              int64_t m, int64_t k, const float* B, int64_t ldb,
                                              int64_t n, float beta, float* C, int64_t ldc,
                                              void* stream) {
    // argument checks, in the same order and with the same codes as spmm_csr_f32
    if (m < 0 || k < 0 || n < 0) return SPMM_ERR_INVALID_ARGUMENT;
    if (m > (int64_t)INT_MAX - BIN_TILE || k > (int64_t)INT_MAX || n > (int64_t)INT_MAX)
        return SPMM_ERR_INVALID_ARGUMENT;
    if (ldb < std::max<int64_t>(1, n) || ldc < std::max<int64_t>(1, n))
        return SPMM_ERR_DIMENSION_MISMATCH;
    if (ldb > (int64_t)INT_MAX) return SPMM_ERR_INVALID_ARGUMENT;   // 32-bit gather offsets
    if (m > NOALLOC_MAX_ROWS || n > NOALLOC_MAX_COLS) return SPMM_ERR_TOO_LARGE;
    if (m == 0 || n == 0) return SPMM_OK;
    if (!C) return SPMM_ERR_NULL_POINTER;
    const bool uses_a = alpha != 0.0f && k > 0;
    if (uses_a && (!row_ptr || !col_idx || !values || !B)) return SPMM_ERR_NULL_POINTER;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SPMM_ERR_CUDA;
    }
    DeviceSetup* ds = nullptr;
    spmm_status_t s = setup_device(dev, &ds);
    if (s != SPMM_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    if (!uses_a)
        return launch_scale<float>(C, ldc, (int)m, (int)n, beta, ds->num_sms * 8, st) == cudaSuccess
                   ? SPMM_OK : SPMM_ERR_CUDA;

    // the handle path's plan (the same geometry, panels and bin thresholds),
    // so the two entry points bin and sum every row alike
    const bool vec = aligned16(B) && aligned16(C) && ldb % 4 == 0 && ldc % 4 == 0;
    const ProductPlan P = plan_product(ds->l2_bytes, k, n, (int)sizeof(float), vec);
    const Geometry geo = P.geo;
    const int long_grid = long_grid_for(ds->num_sms);     // <= NOALLOC_LONG_GRID_MAX (set-up)
    if (m <= SMALL_ROWS) {                // one launch, no scratch (as spmm_csr_f32 does)
        SpmmParams<float> p{};
        p.row_ptr = row_ptr;
        p.col_idx = col_idx;
        p.values = values;
        p.B = B;
        p.ldb = ldb;
        p.C = C;
        p.ldc = ldc;
        p.m = (int)m;
        p.n = (int)n;
        p.alpha = alpha;
        p.beta = beta;
        p.panel_cols = P.panel_cols;
        p.npanels = P.npanels;
        return launch_small<float>(p, geo, P.short_max, ds->num_sms, st) == cudaSuccess
                   ? SPMM_OK : SPMM_ERR_CUDA;
    }

    BinScratch bs{};
    bs.hdr = reinterpret_cast<int*>(ds->scratch + OFF_HDR);
    bs.tile_counts = reinterpret_cast<int*>(ds->scratch + OFF_TILE_COUNTS);
    bs.tile_offsets = reinterpret_cast<int*>(ds->scratch + OFF_TILE_OFFSETS);
    bs.rowlist = reinterpret_cast<int*>(ds->scratch + OFF_ROWLIST);
    bs.med_pre = reinterpret_cast<int*>(ds->scratch + OFF_MED_PRE);
    bs.long_cnt = reinterpret_cast<int*>(ds->scratch + OFF_LONG_CNT);
    bs.long_pre = reinterpret_cast<int*>(ds->scratch + OFF_LONG_PRE);
    bin_geometry(m, &bs.items, &bs.tiles);
    if (launch_binning(row_ptr, (int)m, P.short_max, P.long_min, bs, st, SPMM_PDL) !=
        cudaSuccess)
        return SPMM_ERR_CUDA;

    SpmmParams<float> p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.values = values;
    p.B = B;
    p.ldb = ldb;
    p.C = C;
    p.ldc = ldc;
    p.m = (int)m;
    p.n = (int)n;
    p.alpha = alpha;
    p.beta = beta;
    p.panel_cols = P.panel_cols;
    p.npanels = P.npanels;
    p.rowlist = bs.rowlist;
    p.med_pre = bs.med_pre;
    p.long_cnt = bs.long_cnt;
    p.long_pre = bs.long_pre;
    p.hdr = bs.hdr;
    p.partials = reinterpret_cast<float*>(ds->scratch + OFF_PARTIALS);
    p.long_grid = long_grid;
    const int grid = rows_blocks(ds, geo) * ds->num_sms;
    if (launch_rows<float>(p, geo, grid, st, SPMM_PDL) != cudaSuccess) return SPMM_ERR_CUDA;
    if (launch_long<float>(p, geo, st, SPMM_PDL) != cudaSuccess) return SPMM_ERR_CUDA;
    return SPMM_OK;
}

static_assert(NOALLOC_BYTES < 11u * 1024 * 1024, "static scratch grew past its stated size");
