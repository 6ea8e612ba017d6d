// Internal interfaces between the host driver (spmm_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace spmm {

constexpr unsigned FULL = 0xffffffffu;

// Row bins produced by the pre-pass.  A row of length len goes to
//   SHORT  if len <= short_max   (one lane group per row)
//   MEDIUM if len <  long_min    (one warp per row)
//   LONG   otherwise             (split across CTAs, partial sums + fixup)
enum Bin { BIN_SHORT = 0, BIN_MEDIUM = 1, BIN_LONG = 2, NUM_BINS = 3 };

// Device header written by the pre-pass (int32 words).
enum HeaderWord {
    HDR_COUNT_SHORT = 0,
    HDR_COUNT_MEDIUM = 1,
    HDR_COUNT_LONG = 2,
    HDR_LONG_NNZ = 3,   // total entries in long rows
    HDR_MED_NNZ = 4,    // total entries in medium rows
    HDR_WORDS = 8
};

// Pre-pass geometry: 256 threads; tiles of 512 rows, or one CTA for m <= 2048.
constexpr int BIN_THREADS = 256;
constexpr int BIN_ITEMS = 2;                            // fewest rows per thread, many-tile path
constexpr int BIN_TILE = BIN_THREADS * BIN_ITEMS;       // smallest tile (bounds the tile count)
constexpr int BIN_WAVE_TILES = 1216;                    // tiles kept within about one wave
constexpr int BIN_SINGLE_ITEMS = 8;                     // rows per thread, one-CTA path
constexpr int BIN_SINGLE_ROWS = BIN_THREADS * BIN_SINGLE_ITEMS;   // m up to this: one launch
constexpr int BIN_REC = 8;    // int32 words per tile record

// Products of at most SMALL_ROWS rows run as one launch (small_kernel: every
// CTA bins the rows itself in shared memory).
constexpr int SMALL_ROWS = 2048;

// Long-row kernel geometry.
constexpr int LONG_THREADS = 256;
constexpr int LONG_WARPS = LONG_THREADS / 32;
constexpr int LONG_MIN_SEGMENT = 2048;   // smallest per-CTA share of long-row entries

// Programmatic dependent launch between the kernels of one call.
#ifndef SPMM_PDL
#define SPMM_PDL 1
#endif

// Rows kernel block size and minimum resident blocks per SM (a register cap),
// per geometry.  One block (or two) holds all the SM's resident warps, so the
// warps that interleave over a block's contiguous range of rows are all the
// warps of the SM: rows next to each other in the list, which often gather
// the same B rows, share one L1.  Measured on GB300 against 256-thread blocks
// at the same occupancy: wide-N -3%, Laplacian -2.5%, a SEACells matrix in
// breadth-first row order -5%, the rest unchanged.
#ifndef SPMM_ROWS_THREADS
#define SPMM_ROWS_THREADS 1024
#endif
#ifndef SPMM_ROWS_MIN_BLOCKS
#define SPMM_ROWS_MIN_BLOCKS 1
#endif
#ifndef SPMM_ROWS_THREADS_F64
#define SPMM_ROWS_THREADS_F64 768
#endif
#ifndef SPMM_ROWS_MIN_BLOCKS_F64
#define SPMM_ROWS_MIN_BLOCKS_F64 2
#endif
// binary32 rows kernels with 16-byte vectors and lane groups narrower than a
// warp (n <= 64 columns per panel): twice the gathers in flight per lane, at
// a quarter fewer resident warps (measured faster on power-law and wide-N
// inputs)
#ifndef SPMM_ROWS_THREADS_NARROW
#define SPMM_ROWS_THREADS_NARROW 768
#endif
#ifndef SPMM_ROWS_MIN_BLOCKS_NARROW
#define SPMM_ROWS_MIN_BLOCKS_NARROW 1
#endif
// B bytes each lane keeps in flight per gather batch, and the batch cap.
#ifndef SPMM_BATCH_BYTES
#define SPMM_BATCH_BYTES 64
#endif
#ifndef SPMM_BATCH_BYTES_NARROW
#define SPMM_BATCH_BYTES_NARROW 128
#endif
#ifndef SPMM_BATCH_BYTES_F64
#define SPMM_BATCH_BYTES_F64 16
#endif
#ifndef SPMM_LONG_BATCH_BYTES
#define SPMM_LONG_BATCH_BYTES 64
#endif
#ifndef SPMM_LONG_MIN_BLOCKS
#define SPMM_LONG_MIN_BLOCKS 4
#endif
#ifndef SPMM_BATCH_MAX
#define SPMM_BATCH_MAX 8
#endif

// Rows per thread (2, 4 or 8) and tile count of the many-tile pre-pass for m
// rows: the smallest tiles that keep the count within about one wave.
inline void bin_geometry(int64_t m, int* items, int* tiles) {
    int it = BIN_ITEMS;
    while (it < 8 && (m + BIN_THREADS * it - 1) / (BIN_THREADS * it) > BIN_WAVE_TILES) it *= 2;
    *items = it;
    *tiles = (int)((m + BIN_THREADS * it - 1) / (BIN_THREADS * it));
}

// Kernel launches of the pre-pass for m rows (spmm_bin.cu): one CTA for
// m <= BIN_SINGLE_ROWS; count + scatter while the tiles fit one wave; count +
// scan + scatter beyond.
inline int binning_launches(int64_t m) {
    if (m <= BIN_SINGLE_ROWS) return 1;
    int items, tiles;
    bin_geometry(m, &items, &tiles);
    return tiles <= BIN_WAVE_TILES ? 2 : 3;
}

struct BinScratch {
    int* rowlist;       // [m]  short rows, then medium rows, then long rows (each ascending)
    int* med_pre;       // [m + 1] exclusive prefix of medium-row lengths (stable order)
    int* long_pre;      // [m + 1] exclusive prefix of long-row lengths (stable order)
    int* long_cnt;      // [m] per long row: CTAs that have added their partial (zeroed here)
    int* tile_counts;   // [tiles * BIN_REC] per tile: bin counts, long nnz, medium nnz
    int* tile_offsets;  // [tiles * BIN_REC] exclusive scans of the above over tiles
    int* hdr;           // [HDR_WORDS]
    int tiles;          // many-tile path: tiles of BIN_THREADS * items rows
    int items;
};

template <typename T>
struct SpmmParams {
    const int* row_ptr;
    const int* col_idx;
    const T* values;
    const T* B;
    int64_t ldb;
    T* C;
    int64_t ldc;
    int m;
    int n;               // total columns
    T alpha;
    T beta;
    int keep_c;          // store C with the default L2 policy (a chain reads it next)
    int panel_cols;      // columns per L2 panel (multiple of the vector width)
    int npanels;
    // bins
    const int* rowlist;
    const int* med_pre;
    const int* long_pre;
    int* long_cnt;
    const int* hdr;
    // long-row partial sums: [2 * long_grid, n]
    T* partials;
    int long_grid;
};

// Kernel geometry chosen on the host for one call.
struct Geometry {
    int W;        // elements per vector access (1, 2, 4 or 8)
    int G;        // lanes per row group (power of two <= 32)
    int R;        // vector slots per lane per column pass (1..4)
    bool whole;   // n % W == 0: no lane holds a partial vector
};

// An L2 access-policy window for one launch: accesses to [base, base + bytes)
// are marked persisting with probability hit_ratio (the rest are normal).
struct L2Window {
    const void* base;
    size_t bytes;
    float hit_ratio;
};

// Geometry, column panels and bin thresholds of one product, chosen on the
// host from the operands' shape and alignment and the device's L2 size
// (spmm_api.cu).  Every entry point that launches the product takes its plan
// from here, so equal inputs are binned and summed the same way everywhere.
struct ProductPlan {
    Geometry geo;
    int panel_cols;   // columns per L2 panel of B / C
    int npanels;
    int short_max;    // longest row of the short bin
    int long_min;     // shortest row of the long bin
};
ProductPlan plan_product(int64_t l2_bytes, int64_t k, int64_t n, int es, bool vec);
// CTAs of the long-row launch on a device with num_sms SMs.
int long_grid_for(int num_sms);

// ---- pre-pass (spmm_bin.cu) ----
// `overlap`: launch the dependent kernels of the chain with programmatic
// dependent launch (the first kernel of a call always waits for the stream).
cudaError_t launch_binning(const int* row_ptr, int m, int short_max, int long_min,
                           const BinScratch& s, cudaStream_t st, bool overlap);

// ---- per-bin kernels (spmm_rows_*.cu, spmm_long_*.cu) ----
template <typename T>
cudaError_t launch_rows(const SpmmParams<T>& p, const Geometry& g, int grid, cudaStream_t st,
                        bool overlap, const L2Window* win = nullptr);
template <typename T>
cudaError_t launch_long(const SpmmParams<T>& p, const Geometry& g, cudaStream_t st, bool overlap,
                        const L2Window* win = nullptr);
// m <= SMALL_ROWS: the whole product in one launch (spmm_small_*.cu); p needs
// no bins.  short_max: the short-row threshold of the product's plan.
template <typename T>
cudaError_t launch_small(const SpmmParams<T>& p, const Geometry& g, int short_max, int grid,
                         cudaStream_t st, const L2Window* win = nullptr);

// ---- epilogue-only and checking kernels (spmm_misc.cu) ----
template <typename T>
cudaError_t launch_scale(T* C, int64_t ldc, int m, int n, T beta, int grid, cudaStream_t st);
cudaError_t launch_csr_check(const int* row_ptr, const int* col_idx, int64_t m, int64_t k,
                             int64_t nnz, int* status, cudaStream_t st);
// Binary64 FMA throughput probe: `grid` blocks of 256 threads, grid * 256
// doubles of sink; *fmas receives the FMA instructions one launch executes.
cudaError_t launch_fp64_fma_probe(int grid, int iters, double* sink, cudaStream_t st,
                                  int64_t* fmas);

// Blocks per SM the rows kernel reaches for this geometry (occupancy query).
template <typename T>
int rows_blocks_per_sm(const Geometry& g);

// Host: row_ptr[0] == 0 and non-decreasing (m + 1 entries).
bool csr_rows_valid(const int32_t* row_ptr, int64_t m);
// Host: breadth-first order of the rows of A's pattern (spmm_order.cu).
void row_order_bfs(const int32_t* row_ptr, const int32_t* col_idx, int m, int32_t* order);

}  // namespace spmm

namespace spmm {

// Programmatic dependent launch: a kernel of the chain may be launched while
// its predecessor drains; it waits here before touching the predecessor's
// output (a no-op when launched without the attribute).
__device__ __forceinline__ void wait_for_predecessor() {
#if defined(__CUDA_ARCH__)
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
// Let the next kernel of the chain be scheduled now.
__device__ __forceinline__ void allow_successor() {
#if defined(__CUDA_ARCH__)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Launch `kernel` on `st`, overlapping its launch with the previous kernel
// of the stream when `overlap` is set, with an L2 access-policy window on
// this launch alone when `win` is given (the stream's attributes are left
// untouched).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_windowed(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t st, bool overlap, const L2Window* win,
                                   Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (overlap) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (win && win->bytes > 0) {
        attr[n].id = cudaLaunchAttributeAccessPolicyWindow;
        attr[n].val.accessPolicyWindow.base_ptr = const_cast<void*>(win->base);
        attr[n].val.accessPolicyWindow.num_bytes = win->bytes;
        attr[n].val.accessPolicyWindow.hitRatio = win->hit_ratio;
        attr[n].val.accessPolicyWindow.hitProp = cudaAccessPropertyPersisting;
        attr[n].val.accessPolicyWindow.missProp = cudaAccessPropertyNormal;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t st, bool overlap, Args... args) {
    return launch_windowed(kernel, grid, block, smem, st, overlap, nullptr, args...);
}

}  // namespace spmm
