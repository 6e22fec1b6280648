// gdn_prefill_noalloc: the prefill entry point for callers that cannot
// allocate device memory.
//
// gdn_prefill takes its optional row-order scratch from the caller.  Some
// callers have no way to provide it: code that runs where cudaMalloc is not
// allowed or not wise (an embedding runtime that owns every byte of device
// memory through its own pool, a latency-critical loop where an allocation
// would synchronise the device, a host language binding with no device
// allocator at all).  This variant keeps that scratch in a fixed array that
// lives in the library's own device memory, so the caller passes only inputs
// and outputs.
//
// Every GPU that loads the library holds the array (32 KiB) until the process
// exits.  The array is too small for the per-chunk images of the two-pass
// chunked form, so chunk = 64 always runs the single pass here: the same
// results, but slower than gdn_prefill with its full workspace when the batch
// has fewer heads than the GPU has SMs.  All calls share it: two calls whose work overlaps on the GPU (on
// different streams, or from different host threads) race on it and must be
// ordered by the caller.  Each call writes all of the scratch it reads before
// reading it, so nothing has to be cleared between calls.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace gdn {
namespace {

constexpr size_t kNoAllocScratchBytes = 32768;   // the row order of up to GDN_NOALLOC_MAX_ROWS rows

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once
// per device (in host code the array's name is not a device address).  The
// address is cached for the life of the process; a device reset between calls
// would leave it stale, which the header states is not supported.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace gdn

extern "C" {

gdn_status gdn_prefill_noalloc(const gdn_dims *dims, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const float *g, const float *beta, const float *state_in, float *state_out,
                               const uint8_t *mask, uint16_t *y, int chunk, gdn_stream stream) {
    if (dims == nullptr) return GDN_ERR_INVALID_ARG;
    if (dims->B > GDN_NOALLOC_MAX_ROWS) return GDN_ERR_UNSUPPORTED;
    gdn::Sizes s{dims->B < 0 ? 0 : dims->B, 1, 1, 1, 32, 32, 4, 0.0f};
    if (gdn::row_order_workspace(s) > gdn::kNoAllocScratchBytes) return GDN_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const cudaError_t e = gdn::scratch_address(&scratch);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    return gdn_prefill(dims, q, k, v, g, beta, state_in, state_out, mask, y, chunk, scratch,
                       gdn::kNoAllocScratchBytes, stream);
}

}  // extern "C"
