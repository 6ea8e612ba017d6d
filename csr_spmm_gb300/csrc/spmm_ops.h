// Internal interfaces of the operations beyond the product (the Frank-Wolfe
// gradient scan and ILU(0)) between the host driver (spmm_api.cu) and their
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace spmm {

// ---- Frank-Wolfe gradient scan (spmm_fw.cu) ----
// G = K2B t1 - T2 (n x k), per-column minimum over rows (lowest row on ties),
// gap = sum of B * G over B's stored entries.
template <typename T>
struct FwParams {
    int n, k;
    int ldk;                        // leading dimension of the dense t1 (multiple of FW_TILE)
    const int* k2b_rp; const int* k2b_ci; const T* k2b_v;     // n x k CSR
    const int* t1_rp;  const int* t1_ci;  const T* t1_v;      // k x k CSR
    const int* t2_rp;  const int* t2_ci;  const T* t2_v;      // n x k CSR
    const int* b_rp;   const int* b_ci;   const T* b_v;       // n x k CSR
    T* t1d;                          // scratch: dense t1 [k, ldk], zero padded
    T* part_val;                     // scratch: per-block minima [nblocks, ldk]
    int* part_idx;                   // scratch: per-block argmins [nblocks, ldk]
    double* part_gap;                // scratch: per-block gap sums [nblocks]
    int nwarps;                      // the scan's grid, in warps
    int nblocks;                     // the scan's grid, in blocks
    T* out_val;                      // [k]
    int* out_idx;                    // [k]
    T* out_gap;                      // [1]
};
constexpr int FW_THREADS = 256;
// columns per pass of a warp: 32 lanes x one 16-byte vector
template <typename T> constexpr int fw_tile() { return 32 * (16 / (int)sizeof(T)); }
template <typename T>
cudaError_t launch_fw(const FwParams<T>& p, int grid, cudaStream_t st);
template <typename T>
int fw_blocks_per_sm(int k);

// ---- ILU(0), dataflow-scheduled (spmm_ilu0.cu) ----
template <typename T>
struct Ilu0Params {
    int n;
    int64_t nnz;
    const int* rp;
    const int* ci;
    T* v;                  // A's values in, the L \ U factors out (in place)
    int* depth;            // optional: each row's level
    // scratch
    int* pending;          // [n] lower entries of the row not yet final
    int* cnt;              // [n] rows depending on the row (then a fill cursor)
    int* dep_ptr;          // [n + 1] start of each row's dependents
    int* dep_idx;          // [nnz] dependent rows, grouped by the row they depend on
    int2* piv;             // [nnz] per lower entry (i, k): the position of a_kk in row k
                           //       (-1: none) and the end of row k
    int4* rec;             // [n * ILU0_REC_LANES] per-row structure records (ilu0_records)
    int* tile_sum;         // [ceil(n / 1024)] tile sums, then tile offsets, of the dependent counts
    T* pub;                // [nnz] published final values (the sentinel until written)
    int* done;             // [n] 1: a value the row published is the sentinel's bit pattern
    int* queue;            // [n] rows in the order they became ready (-1: not yet)
    int* head;             // next queue slot to take
    int* tail;             // next queue slot to fill
    int* abort;            // stop every warp (a failure was met)
    int* finished;         // rows factored so far (termination and progress)
    int* status;           // caller's: 0, or ILU0 failure bits
};
// Factorisation block, one per SM: four warps (the 707 x 707 Laplacian in
// binary64 on GB300: 5.01 ms with 128 threads, 5.04 with 192, 5.06 with 256,
// 5.10 with 384, 5.31 with 512: fewer idle warps polling the queue; but
// 5.19 with 96 and 6.21 with 64, too few warps for the widest levels).
#ifndef SPMM_ILU0_THREADS
#define SPMM_ILU0_THREADS 128
#endif
constexpr int ILU0_THREADS = SPMM_ILU0_THREADS;
// A row's structure record: ILU0_REC_LANES int4 words, lane q holding
// {column of entry q, pivot position and end of row k for a lower entry q,
// dependent q}; lane 14's last word is the row's first entry, lane 15's its
// length | dependents << 8 (or -1: too long for a record).
constexpr int ILU0_REC_LANES = 16;
template <typename T>
cudaError_t launch_ilu0(const Ilu0Params<T>& p, int grid, cudaStream_t st);
template <typename T>
int ilu0_blocks_per_sm();

}  // namespace spmm
