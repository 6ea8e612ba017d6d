// Row order for locality (host code).
//
// The rows kernel hands each block a contiguous range of a row list, and the
// block's warps walk that range together.  When rows that sit next to each
// other in the list gather the same B rows, those gathers are served by the
// SM's L1 instead of crossing to L2.  A kernel matrix built from a k-nearest-
// neighbour graph (the SEACells kernel of the bixverse page) has that
// structure, but its row numbering rarely shows it.  A breadth-first
// traversal of the graph of A's pattern puts neighbours next to each other.
//
// Graph: vertex i is row i; row i has an edge to row j for every stored entry
// (i, j) with 0 <= j < m.  Entries in columns outside [0, m) are skipped
// (they name no row).  The traversal starts at row 0, visits the neighbours of
// each row in stored order, and when a component is exhausted it starts again
// at the lowest unvisited row, so every row appears exactly once.  This is
// the Cuthill-McKee traversal without its sort of neighbours by degree
// (measured on GB300: the degree sort makes no difference to the product).
#include <climits>
#include <cstdint>
#include <new>
#include <vector>

#include "csr_spmm.h"
#include "spmm_internal.h"

namespace spmm {

bool csr_rows_valid(const int32_t* row_ptr, int64_t m) {
    if (row_ptr[0] != 0) return false;
    for (int64_t i = 0; i < m; ++i)
        if (row_ptr[i + 1] < row_ptr[i]) return false;
    return true;
}

void row_order_bfs(const int32_t* row_ptr, const int32_t* col_idx, int m, int32_t* order) {
    std::vector<unsigned char> seen((size_t)m, 0);
    int head = 0, tail = 0;                       // order[head..tail) is the queue
    for (int root = 0; root < m; ++root) {
        if (seen[root]) continue;
        seen[root] = 1;
        order[tail++] = root;
        while (head < tail) {
            const int r = order[head++];
            for (int32_t p = row_ptr[r]; p < row_ptr[r + 1]; ++p) {
                const int32_t c = col_idx[p];
                if (c >= 0 && c < m && !seen[c]) {
                    seen[c] = 1;
                    order[tail++] = c;
                }
            }
        }
    }
}

}  // namespace spmm

extern "C" spmm_status_t spmm_row_order_bfs(const int32_t* row_ptr, const int32_t* col_idx,
                                            int64_t m, int32_t* order) {
    if (m < 0 || m > (int64_t)INT_MAX - 1) return SPMM_ERR_INVALID_ARGUMENT;
    if (m == 0) return SPMM_OK;
    if (!row_ptr || !order) return SPMM_ERR_NULL_POINTER;
    if (!spmm::csr_rows_valid(row_ptr, m)) return SPMM_ERR_INVALID_CSR;
    if (row_ptr[m] > 0 && !col_idx) return SPMM_ERR_NULL_POINTER;
    try {
        spmm::row_order_bfs(row_ptr, col_idx, (int)m, order);
    } catch (const std::bad_alloc&) {          // no C++ exception crosses the C ABI
        return SPMM_ERR_ALLOC;
    }
    return SPMM_OK;
}
