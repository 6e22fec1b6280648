// Self-test of the failure path: a wait that runs out is reported, and the
// context stays usable.  One thread initialises an mbarrier that nothing ever
// arrives on, waits on it with a short iteration limit (the same bounded
// try_wait loop the kernels use, with a smaller limit), and on expiry sets
// the device error word like any kernel whose wait gives up.  No fault, trap
// or unbounded wait is involved.
#include "common.cuh"
#include "internal.h"

namespace gdn {
namespace {

constexpr uint32_t kSelftestSpins = 1u << 12;

__global__ void wait_timeout_kernel(unsigned *err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    for (uint32_t i = 0; i < kSelftestSpins; ++i)
        if (mbar_try_wait(&bar, 0)) return;   // never completes: nothing arrives
    atomicOr(err, kErrMbarTimeout);
}

}  // namespace

cudaError_t launch_selftest_timeout(unsigned *err, cudaStream_t st) {
    wait_timeout_kernel<<<1, 32, 0, st>>>(err);
    return cudaGetLastError();
}

}  // namespace gdn
