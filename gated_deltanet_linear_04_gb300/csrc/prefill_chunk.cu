// Chunked (WY / UT-transform) prefill on the tensor cores.
#include "common.cuh"
#include "internal.h"

namespace gdn {

size_t prefill_chunked_workspace(const Sizes &) { return 0; }

cudaError_t launch_prefill_chunked(const Sizes &, const uint16_t *, const uint16_t *, const uint16_t *,
                                   const float *, const float *, const float *, float *, const uint8_t *,
                                   uint16_t *, void *, unsigned *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace gdn
