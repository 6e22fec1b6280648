// Host-side launchers of the GB300 kernels (one translation unit each), called
// by the C ABI in api.cu after argument validation.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

struct Sizes {
    int B, T, Hk, Hv, Dk, Dv, K;
    float eps;
    int C() const { return 2 * Hk * Dk + Hv * Dv; }
};

int num_sms();  // SMs of the current device (cached per device)

// Kernel attributes (dynamic shared memory, cluster size) belong to the
// device context that was current when they were set, so a launcher applies
// them once per device: `done` holds one bit per device ordinal (0..63; a
// higher ordinal is set on every call).  Concurrent first calls may both run
// `apply`, which is harmless.
template <typename F>
cudaError_t once_per_device(unsigned long long &done, F &&apply) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit != 0ull && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) & bit) != 0ull) return cudaSuccess;
    e = apply();
    if (e == cudaSuccess && bit != 0ull) __atomic_fetch_or(&done, bit, __ATOMIC_RELEASE);
    return e;
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device.
template <typename K>
cudaError_t set_max_smem(unsigned long long &done, K kernel, size_t bytes) {
    return once_per_device(done, [&] {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    });
}

cudaError_t launch_conv_update(const Sizes &s, const uint16_t *qkv, const uint16_t *conv_w, uint16_t *conv_state,
                               const uint8_t *mask, uint16_t *q, uint16_t *k, uint16_t *v, unsigned *err,
                               cudaStream_t st);

cudaError_t launch_gating(const Sizes &s, const uint16_t *a, const uint16_t *b, const float *A_log,
                          const float *dt_bias, float *g, float *beta, cudaStream_t st);

cudaError_t launch_decode(const Sizes &s, const uint16_t *qkv, const uint16_t *conv_w, uint16_t *conv_state,
                          const uint16_t *a, const uint16_t *b, const float *A_log, const float *dt_bias,
                          float *state, const uint8_t *row_mask, uint16_t *y, const uint16_t *z,
                          const float *norm_w, float norm_eps, unsigned *err, cudaStream_t st);

cudaError_t launch_decode_window(const Sizes &s, const uint16_t *qkv, const uint16_t *conv_w, uint16_t *conv_state,
                                 const uint16_t *a, const uint16_t *b, const float *A_log, const float *dt_bias,
                                 float *state, const int32_t *keep, uint16_t *y, unsigned *err, cudaStream_t st);

// Encodes a 3-D row-major tensor map (d2 x d1 x d0, d0 innermost; box
// box1 x box0 in the two inner dimensions, one deep in the outer), no swizzle.
bool encode_tmap_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes, uint64_t d2,
                    uint64_t d1, uint64_t d0, uint32_t box1, uint32_t box0);

// Encodes a dense row-major tensor map of `rank` dimensions (dims and box
// innermost first).  A box may be wider than its dimension: the elements past
// the end read as zeros (loads) or are not written (stores).
bool encode_tmap(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes, int rank,
                 const uint64_t *dims, const uint32_t *box, CUtensorMapSwizzle swizzle);

// Encodes a 2-D row-major tensor map (rows x cols, box rows x box_cols).
bool encode_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                    uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols,
                    CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE);

// Row order for masked prefill (row_order.cu): order[i] = the row the i-th
// row slot of a prefill launch processes, longest (most chunks holding a
// valid step) first.  Scratch: row_order_workspace(s) bytes, order at offset 0.
size_t row_order_workspace(const Sizes &s);
cudaError_t launch_row_order(const Sizes &s, const uint8_t *mask, void *ws, cudaStream_t st);

// `order` (optional, with a mask): row slot -> batch row, see above.
cudaError_t launch_prefill_seq(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const float *g, const float *beta, const float *state_in, float *state_out,
                               const uint8_t *mask, const int *order, uint16_t *y, unsigned *err,
                               cudaStream_t st);

cudaError_t launch_rmsnorm_gated(const Sizes &s, const uint16_t *y, const uint16_t *z, const float *norm_w,
                                 float eps, uint16_t *out, cudaStream_t st);

cudaError_t launch_prefill_seq_vec(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                   const float *g_vec, const float *beta, const float *state_in, float *state_out,
                                   const uint8_t *mask, uint16_t *y, unsigned *err, cudaStream_t st);

cudaError_t launch_prefill_chunked(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                   const float *g, const float *beta, const float *state_in, float *state_out,
                                   const uint8_t *mask, const int *order, uint16_t *y, const uint16_t *z,
                                   const float *norm_w, float norm_eps, unsigned *err, cudaStream_t st,
                                   float *rec_s = nullptr, float *rec_d = nullptr);

// Failure-path self-test (selftest.cu): a kernel whose bounded wait runs out.
cudaError_t launch_selftest_timeout(unsigned *err, cudaStream_t st);

// Backward pass (backward.cu): workspace bytes and the launch (outputs zeroed
// by the launch, then accumulated).
size_t backward_workspace(const Sizes &s);
cudaError_t launch_backward(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const float *g, const float *beta, const float *state_in, const uint8_t *mask,
                            const uint16_t *dy, const float *dstate_out, float *dq, float *dk, float *dv,
                            float *dg, float *dbeta, float *dstate_in, void *ws, cudaStream_t st);

// Two-pass chunked form (prefill_chunk2.cu) for batches with fewer heads than
// SMs: bytes of its workspace blobs, whether it is the faster form for these
// sizes, and the launch (blobs: 16-byte aligned, prefill_two_pass_workspace
// bytes).
size_t prefill_two_pass_workspace(const Sizes &s);
bool prefill_two_pass_pays(const Sizes &s);
cudaError_t launch_prefill_two_pass(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                    const float *g, const float *beta, const float *state_in, float *state_out,
                                    const uint8_t *mask, const int *order, uint16_t *y, void *blobs,
                                    unsigned *err, cudaStream_t st, float *rec_s = nullptr,
                                    float *rec_d = nullptr);

// Chunked backward (backward_chunk.cu, Dk = Dv = 128): workspace bytes and the
// launch (outputs zeroed by the launch, then written or accumulated).  The
// forward's records (rec_s, rec_d above) are taken by the chunked forward
// kernels on the way.
size_t backward_chunked_workspace(const Sizes &s);
cudaError_t launch_backward_chunked(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                    const float *g, const float *beta, const float *state_in, const uint8_t *mask,
                                    const uint16_t *dy, const float *dstate_out, float *dq, float *dk, float *dv,
                                    float *dg, float *dbeta, float *dstate_in, void *ws, unsigned *err,
                                    cudaStream_t st);

}  // namespace gdn
