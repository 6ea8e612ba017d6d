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
constexpr int NOALLOC_LONG_GRID_MAX = 640;         // 4 CTAs per SM for up to 160 SMs

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
        s.supported = (major == 10 && minor == 3);
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

inline int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
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

    // plan: vector width, one column panel (n <= 512 keeps k x n panels of
    // small problems whole), lane groups, bin thresholds -- the same rules the
    // handle path applies
    struct Shape { Geometry geo; int panel_cols; };
    auto shape_for = [&](int W) {
        Shape sh{};
        sh.geo.W = W;
        int64_t panel = n;
        const double bbytes = (double)k * (double)n * sizeof(float);
        if (ds->l2_bytes > 0 && bbytes > 3.0 * (double)ds->l2_bytes) {
            const int64_t align = std::max<int64_t>(W, 32);
            int64_t cols = (int64_t)(0.5 * (double)ds->l2_bytes / ((double)k * sizeof(float)));
            cols = cols / align * align;
            if (cols < align) cols = align;
            const int64_t np = (n + cols - 1) / cols;
            panel = (n + np - 1) / np;
            panel = (panel + W - 1) / W * W;
        }
        sh.panel_cols = (int)std::min<int64_t>(panel, n);
        const int nvec = (sh.panel_cols + W - 1) / W;
        if (nvec <= 32) {
            sh.geo.G = next_pow2(nvec);
            sh.geo.R = 1;
        } else {
            sh.geo.G = 32;
            sh.geo.R = nvec <= 64 ? 2 : 4;
        }
        return sh;
    };
    const bool vec = aligned16(B) && aligned16(C) && ldb % 4 == 0 && ldc % 4 == 0;
    const Shape sh = shape_for(vec ? 4 : 1);
    const Geometry geo = sh.geo;
    const int panel_cols = sh.panel_cols;
    const int npanels = (int)((n + panel_cols - 1) / panel_cols);
    // bin thresholds from the 16-byte geometry whatever the alignment (the
    // bins then depend only on row lengths and n, as on the handle path)
    const Geometry g16 = vec ? geo : shape_for(4).geo;
    const int bytes_per_entry = g16.R * g16.W * (int)sizeof(float);
    const int U = std::min(SPMM_BATCH_MAX, std::max(1, SPMM_BATCH_BYTES / bytes_per_entry));
    const int CH = std::max(g16.G, U);
    const int long_min = 1024;
    const int short_max = g16.G == 32 ? long_min - 1 : std::min(long_min - 1, 2 * CH);
    const int long_grid = std::min(4 * ds->num_sms, NOALLOC_LONG_GRID_MAX);

    BinScratch bs{};
    bs.hdr = reinterpret_cast<int*>(ds->scratch + OFF_HDR);
    bs.tile_counts = reinterpret_cast<int*>(ds->scratch + OFF_TILE_COUNTS);
    bs.tile_offsets = reinterpret_cast<int*>(ds->scratch + OFF_TILE_OFFSETS);
    bs.rowlist = reinterpret_cast<int*>(ds->scratch + OFF_ROWLIST);
    bs.med_pre = reinterpret_cast<int*>(ds->scratch + OFF_MED_PRE);
    bs.long_cnt = reinterpret_cast<int*>(ds->scratch + OFF_LONG_CNT);
    bs.long_pre = reinterpret_cast<int*>(ds->scratch + OFF_LONG_PRE);
    bin_geometry(m, &bs.items, &bs.tiles);
    if (launch_binning(row_ptr, (int)m, short_max, long_min, bs, st, SPMM_PDL) != cudaSuccess)
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
    p.panel_cols = panel_cols;
    p.npanels = npanels;
    p.rowlist = bs.rowlist;
    p.med_pre = bs.med_pre;
    p.long_cnt = bs.long_cnt;
    p.long_pre = bs.long_pre;
    p.hdr = bs.hdr;
    p.partials = reinterpret_cast<float*>(ds->scratch + OFF_PARTIALS);
    p.long_grid = long_grid;
    const int grid = rows_blocks_per_sm<float>(geo) * ds->num_sms;
    if (launch_rows<float>(p, geo, grid, st, SPMM_PDL) != cudaSuccess) return SPMM_ERR_CUDA;
    if (launch_long<float>(p, geo, st, SPMM_PDL) != cudaSuccess) return SPMM_ERR_CUDA;
    return SPMM_OK;
}

static_assert(NOALLOC_BYTES < 11u * 1024 * 1024, "static scratch grew past its stated size");
