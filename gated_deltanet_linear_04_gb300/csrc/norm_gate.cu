// RMSNormGated output of the layer: out = bf16( silu(z) * w * y / sqrt(mean(y^2) + eps) )
// over the Dv values of each (b, t, hv) head row ("mlex 0.1.2,
// src/models/gated_delta.rs", GatedDeltaNet::forward: the f32 rms_norm of y,
// the norm weight, the silu(z) gate, the cast back to the activation dtype).
//
// HBM-bound: 2 bytes of y + 2 of z in, 2 out per element.  One warp per head
// row (Dv/32 values per lane, one 2-8 byte load each), four rows per warp
// iteration so that several rows' loads are in flight; the row sum of
// squares is a warp shuffle sum.
#include "common.cuh"
#include "internal.h"

namespace gdn {
namespace {

constexpr int kRowsPerIter = 4;

template <int CPL>
__device__ __forceinline__ void ld_bf16(const uint16_t *p, float (&o)[CPL]) {
    if constexpr (CPL == 4) {
        const uint2 r = *reinterpret_cast<const uint2 *>(p);
        o[0] = __uint_as_float(r.x << 16);
        o[1] = __uint_as_float(r.x & 0xffff0000u);
        o[2] = __uint_as_float(r.y << 16);
        o[3] = __uint_as_float(r.y & 0xffff0000u);
    } else if constexpr (CPL == 2) {
        const uint32_t r = *reinterpret_cast<const uint32_t *>(p);
        o[0] = __uint_as_float(r << 16);
        o[1] = __uint_as_float(r & 0xffff0000u);
    } else {
        o[0] = bf16_to_f32(*p);
    }
}

template <int CPL>
__device__ __forceinline__ void st_bf16(uint16_t *p, const float (&x)[CPL]) {
    if constexpr (CPL == 4) {
        uint2 r;
        r.x = (uint32_t)f32_to_bf16(x[0]) | ((uint32_t)f32_to_bf16(x[1]) << 16);
        r.y = (uint32_t)f32_to_bf16(x[2]) | ((uint32_t)f32_to_bf16(x[3]) << 16);
        *reinterpret_cast<uint2 *>(p) = r;
    } else if constexpr (CPL == 2) {
        *reinterpret_cast<uint32_t *>(p) = (uint32_t)f32_to_bf16(x[0]) | ((uint32_t)f32_to_bf16(x[1]) << 16);
    } else {
        *p = f32_to_bf16(x[0]);
    }
}

template <int DV>
__global__ void __launch_bounds__(256) rmsnorm_gated_kernel(const uint16_t *__restrict__ y,
                                                            const uint16_t *__restrict__ z,
                                                            const float *__restrict__ w, float eps,
                                                            uint16_t *__restrict__ out, size_t rows) {
    constexpr int CPL = DV / 32;
    const int lane = threadIdx.x & 31;
    const size_t warp = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
    float wv[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) wv[i] = w[lane * CPL + i];
    const float inv_d = 1.0f / (float)DV;
    for (size_t r0 = warp * kRowsPerIter; r0 < rows; r0 += nwarps * kRowsPerIter) {
        float yv[kRowsPerIter][CPL], zv[kRowsPerIter][CPL];
#pragma unroll
        for (int k = 0; k < kRowsPerIter; ++k) {
            if (r0 + k < rows) {
                ld_bf16<CPL>(y + (r0 + k) * DV + lane * CPL, yv[k]);
                ld_bf16<CPL>(z + (r0 + k) * DV + lane * CPL, zv[k]);
            } else {
#pragma unroll
                for (int i = 0; i < CPL; ++i) yv[k][i] = zv[k][i] = 0.0f;
            }
        }
#pragma unroll
        for (int k = 0; k < kRowsPerIter; ++k) {
            float ss = 0.0f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) ss = fmaf(yv[k][i], yv[k][i], ss);
            ss = warp_sum(ss);
            const float rs = 1.0f / sqrtf(ss * inv_d + eps);
            float o[CPL];
#pragma unroll
            for (int i = 0; i < CPL; ++i) o[i] = silu(zv[k][i]) * ((yv[k][i] * rs) * wv[i]);
            if (r0 + k < rows) st_bf16<CPL>(out + (r0 + k) * DV + lane * CPL, o);
        }
    }
}

template <int DV>
cudaError_t launch_t(const uint16_t *y, const uint16_t *z, const float *w, float eps, uint16_t *out, size_t rows,
                     cudaStream_t st) {
    const size_t warps = (rows + kRowsPerIter - 1) / kRowsPerIter;
    size_t blocks = (warps + 7) / 8;
    const size_t cap = (size_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    rmsnorm_gated_kernel<DV><<<(unsigned)blocks, 256, 0, st>>>(y, z, w, eps, out, rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm_gated(const Sizes &s, const uint16_t *y, const uint16_t *z, const float *norm_w,
                                 float eps, uint16_t *out, cudaStream_t st) {
    const size_t rows = (size_t)s.B * s.T * s.Hv;
    switch (s.Dv) {
        case 32: return launch_t<32>(y, z, norm_w, eps, out, rows, st);
        case 64: return launch_t<64>(y, z, norm_w, eps, out, rows, st);
        case 128: return launch_t<128>(y, z, norm_w, eps, out, rows, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
