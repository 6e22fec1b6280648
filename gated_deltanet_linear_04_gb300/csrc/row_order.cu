// Longest-first row order for masked prefill.
//
// With right-padded rows of mixed lengths the prefill kernels' cost per row
// is the number of its 64-step chunks that hold a valid step (wholly masked
// chunks are skipped).  Rows are processed by independent CTAs that the
// hardware dispatches in index order as earlier ones finish, so handing the
// longest rows out first (greedy list scheduling in decreasing order of work)
// keeps a long row from starting last and setting the tail of the launch.
// Two small kernels: the work of each row, then each row's rank.  The order
// only decides which CTA takes which row; every row's results are the same.
#include "common.cuh"
#include "internal.h"
#include "mask_scan.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;

// work[b] = number of chunks of row b holding a valid step; one CTA per row
__global__ void __launch_bounds__(kThreads) row_work_kernel(const uint8_t *mask, int T, int *work) {
    const int b = blockIdx.x;
    const uint8_t *mrow = mask + (size_t)b * T;
    const int nch = (T + 63) / 64;
    int n = 0;
    for (int c0 = 0; c0 < nch; c0 += kThreads) {
        const int ch = c0 + (int)threadIdx.x;
        n += __syncthreads_count(ch < nch && chunk_has_valid(mrow, T, ch));
    }
    if (threadIdx.x == 0) work[b] = n;
}

// order[rank(b)] = b, ranks by decreasing work, ties in index order
__global__ void __launch_bounds__(kThreads) row_rank_kernel(const int *work, int B, int *order) {
    const int b = blockIdx.x * kThreads + (int)threadIdx.x;
    if (b >= B) return;
    const int w = work[b];
    int r = 0;
    for (int i = 0; i < B; ++i) {
        const int wi = __ldg(work + i);
        r += (wi > w) || (wi == w && i < b);
    }
    order[r] = b;
}

size_t work_offset(int B) { return ((size_t)B * sizeof(int) + 15) & ~(size_t)15; }

}  // namespace

size_t row_order_workspace(const Sizes &s) {
    if (s.B <= 0) return 0;
    return (work_offset(s.B) + (size_t)s.B * sizeof(int) + 255) & ~(size_t)255;
}

cudaError_t launch_row_order(const Sizes &s, const uint8_t *mask, void *ws, cudaStream_t st) {
    int *order = static_cast<int *>(ws);
    int *work = reinterpret_cast<int *>(static_cast<char *>(ws) + work_offset(s.B));
    row_work_kernel<<<s.B, kThreads, 0, st>>>(mask, s.T, work);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    row_rank_kernel<<<(s.B + kThreads - 1) / kThreads, kThreads, 0, st>>>(work, s.B, order);
    return cudaGetLastError();
}

}  // namespace gdn
