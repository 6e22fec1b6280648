// Device helpers shared by the GB300 kernels: bf16 conversion, warp sums,
// mbarrier / bulk-copy / TMA / cluster-barrier wrappers (inline PTX, sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {

// Error word bits set by kernels whose bounded waits give up.
enum : unsigned {
    kErrMbarTimeout = 1u,
    kErrMmaTimeout = 2u,
};

// Spin limit of every bounded wait: try_wait suspends for a hardware-chosen
// interval per probe, so this is seconds of wall time, far beyond any real
// copy latency, yet finite.
constexpr uint32_t kSpinLimit = 1u << 24;

__device__ __forceinline__ float bf16_to_f32(uint16_t bits) {
    return __uint_as_float(static_cast<uint32_t>(bits) << 16);
}

// Round-to-nearest-even f32 -> bf16 bit pattern.
__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&h);
}

// The value of x after one RNE rounding to bf16, as f32.
__device__ __forceinline__ float round_bf16(float x) { return bf16_to_f32(f32_to_bf16(x)); }

template <int WIDTH = 32>
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// e^x as 2^(x log2 e) on the hardware base-2 exponential unit (ex2.approx,
// relative error ~2^-22; results below 2^-126 flush to zero).
__device__ __forceinline__ float exp_fast(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x * 1.4426950408889634f));
    return r;
}

__device__ __forceinline__ float rcp_fast(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// x * sigmoid(x); its result is rounded to bf16 by every caller, so the
// approximate exponential and reciprocal (each ~1-2 ulp of f32) are invisible
// except where the f32 value sits on a bf16 rounding boundary.  For x -> -inf
// the exponential overflows to inf and the reciprocal gives 0, so the result
// tends to -0 as it should.
__device__ __forceinline__ float silu(float u) { return u * rcp_fast(1.0f + exp_fast(-u)); }

__device__ __forceinline__ float softplus(float x) {
    return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
}

__device__ __forceinline__ float sigmoid(float x) { return 1.0f / (1.0f + expf(-x)); }

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy and the cluster.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns
// false (and sets the error word) if the limit is reached.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned *err) {
    for (uint32_t i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    if (err) atomicOr(err, kErrMbarTimeout);
    return false;
}

// ---------------------------------------------------------------------------
// bulk copies (TMA engine)
// ---------------------------------------------------------------------------
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 1-D bulk copy shared -> global, tracked by the issuing thread's bulk group.
__device__ __forceinline__ void bulk_store(void *gmem_dst, const void *smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ... every committed group but the most recent one
__device__ __forceinline__ void bulk_wait_all_but_newest() {
    asm volatile("cp.async.bulk.wait_group 1;" ::: "memory");
}

// Wait until every committed bulk store has finished reading its shared-memory
// source (the global writes may still be in flight; they complete with the
// grid).  Enough before a CTA exits or reuses the buffer.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy / tensor core) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled TMA load: box at (x = inner coordinate, y = row) of `tmap`.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const void *tmap, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled TMA load: box at (x = inner coordinate, y, z) of `tmap` (x times
// the element size a multiple of 16 bytes; out-of-range rows read as zeros).
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const void *tmap, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// 4-D tiled TMA store of the box at (x, y, z, w) of `tmap` from shared memory,
// tracked by the issuing thread's bulk group (clipped at the tensor's bounds).
__device__ __forceinline__ void tma_store_4d(const void *tmap, int x, int y, int z, int w, const void *smem_src) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(tmap),
                 "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(smem_src))
                 : "memory");
}

// 3-D tiled TMA store of the box at (x = inner coordinate, y, z) of `tmap`
// from shared memory, tracked by the issuing thread's bulk group (the box is
// clipped at the tensor's bounds; x * element size must be a multiple of 16).
__device__ __forceinline__ void tma_store_3d(const void *tmap, int x, int y, int z, const void *smem_src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(tmap),
                 "r"(x), "r"(y), "r"(z), "r"(smem_u32(smem_src))
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Four consecutive f32 added to global memory in one reduction (p 16-byte
// aligned); no return value.
__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Programmatic dependent launch: the next grid on the stream may be scheduled
// as soon as every CTA of this one has called grid_dep_launch; it then waits
// (grid_dep_wait) for the previous grid to finish and its writes to be
// visible before touching any buffer that grid may write.  Both are no-ops
// for a grid launched without the programmatic-serialization attribute.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// thread-block clusters
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// Arrive without release semantics: does not wait for this thread's
// outstanding memory accesses.  Usable when the only accesses that must be
// ordered before the other CTAs' post-wait writes are loads whose values have
// already been consumed (a consumed load has completed).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace gdn
