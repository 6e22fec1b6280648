// Skipping fully masked 64-step chunks in the prefill kernels.
//
// A masked step leaves the recurrent state untouched and writes y = 0 (the
// masked specialization of gated_delta_step in "mlx-bun 0.4.0 -> 1.0.0,
// package/src/model/qwen3-delta.ts"), so a chunk whose 64 steps are all masked
// is the identity on the state: the kernels write its zero outputs and move
// on without staging its inputs.  Right-padded batches of mixed lengths are
// mostly such chunks at the tail of the shorter rows.
//
// The search keeps a bitmap of the chunks that hold at least one valid step
// for a window of NT chunks (thread i tests chunk base + i), in shared memory;
// it is rebuilt when the search leaves the window.  All calls are made by the
// whole block with the same arguments (they contain block barriers).
#pragma once

#include <stdint.h>

namespace gdn {

// True if chunk `ch` (steps [64 ch, min(64 ch + 64, T))) of a mask row holds a
// valid (non-zero) step.
__device__ __forceinline__ bool chunk_has_valid(const uint8_t *mrow, int T, int ch) {
    const int t0 = ch * 64, n = min(64, T - t0);
    const uint8_t *p = mrow + t0;
    if (n == 64 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
        const uint4 *p16 = reinterpret_cast<const uint4 *>(p);
        uint32_t acc = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 w = p16[i];
            acc |= w.x | w.y | w.z | w.w;
        }
        return acc != 0;
    }
    uint32_t acc = 0;
    for (int i = 0; i < n; ++i) acc |= p[i];
    return acc != 0;
}

template <int NT>
struct ChunkScan {
    static_assert(NT % 32 == 0, "window is a whole number of warps");
    static constexpr int kWords = NT / 32;
    static constexpr int kStep = 64;   // steps per chunk

    const uint8_t *mrow;   // mask row of this batch row (nullptr: every step valid)
    int T, nchunks;
    uint32_t *bits;        // shared, kWords words
    int wb;                // first chunk of the scanned window

    __device__ ChunkScan(const uint8_t *mask_row, int T_, uint32_t *shared_bits)
        : mrow(mask_row), T(T_), nchunks((T_ + kStep - 1) / kStep), bits(shared_bits), wb(-(1 << 30)) {}

    __device__ __forceinline__ void scan(int from) {
        __syncthreads();   // every thread is done with the previous window
        const int ch = from + (int)threadIdx.x;
        const bool any = ch < nchunks && chunk_has_valid(mrow, T, ch);
        const unsigned bal = __ballot_sync(0xffffffffu, any);
        if ((threadIdx.x & 31u) == 0) bits[threadIdx.x >> 5] = bal;
        wb = from;
        __syncthreads();
    }

    // Smallest chunk index >= from holding a valid step, else nchunks.
    __device__ __forceinline__ int next_active(int from) {
        if (mrow == nullptr) return min(from, nchunks);
        while (from < nchunks) {
            if (from - wb >= NT) scan(from);
            const int off = from - wb;
            int w = off >> 5;
            uint32_t m = bits[w] & (0xffffffffu << (off & 31));
            while (m == 0u && ++w < kWords) m = bits[w];
            if (m != 0u) return min(wb + w * 32 + __ffs((int)m) - 1, nchunks);
            from = wb + NT;
        }
        return nchunks;
    }
};

// Zero y for steps [t_begin, t_end) of one row: `width` bf16 values per step
// (a multiple of 8) starting at `first` (16-byte aligned), rows `stride`
// elements apart.  Called by the whole block, whose size is a multiple of
// width / 8: each thread keeps one 16-byte column group and steps through
// the rows (plain 16-byte stores, no division in the loop).
__device__ __forceinline__ void zero_y_rows(uint16_t *first, size_t stride, int t_begin, int t_end, int width) {
    const int per = width >> 3;
    const int c8 = (int)(threadIdx.x % (unsigned)per) * 8;
    const int rows_per_pass = (int)blockDim.x / per;
    for (int t = t_begin + (int)(threadIdx.x / (unsigned)per); t < t_end; t += rows_per_pass)
        *reinterpret_cast<uint4 *>(first + (size_t)t * stride + (size_t)c8) = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace gdn
