// Prefill-side elementwise kernels: the fused conv window + depthwise conv +
// SiLU + q/k rms-norm/scale (gdn_conv_update) and the gates (gdn_gating).
//
// Definitions: "mlex 0.1.2, src/models/gated_delta.rs", GatedDeltaNet::forward
// (conv_state concat and slice, conv1d with one group per channel, silu, split
// into q/k/v, rms_norm without weight, q scaled by 1/Dk and k by 1/sqrt(Dk));
// "mlx-bun 0.4.0 -> 1.0.0, package/src/model/qwen3-delta.ts", computeG and the
// masked gated_delta_step (a masked step takes no part in the update).
//
// Work split (memory-bound, ~2 bytes in + 2 bytes out per channel-token): one
// warp owns one head segment (Dk q- or k-channels, or Dv v-channels) for a
// tile of 8 consecutive tokens (four 8-warp CTAs resident per SM).  Each lane
// holds D/32 channels.  All rows of the tile are loaded up front (independent
// loads in flight per lane), then the warp walks the tile in order keeping the
// last K-1 *valid* rows in registers,
// so every qkv element is read once.  The rms-norm is a warp shuffle sum.
//
// Masked steps ("skip" reading): they do not enter the conv window; their q/k/v
// are written as zeros.  The K-1 valid rows preceding a tile are found by a
// warp-ballot scan backwards over the mask; missing rows come from conv_state.
// The new conv_state is written by a second, tiny kernel that runs after the
// first on the stream, because tiles anywhere in the row may still read the
// old conv_state.
#include "common.cuh"
#include "internal.h"

namespace gdn {
namespace {

constexpr int kTile = 8;        // tokens per warp task (8: measured 1.3x faster than 16 at 4 CTAs/SM)
constexpr int kWarps = 8;       // head segments per CTA
constexpr int kMaxHalo = 3;     // K - 1 for the largest supported K (4)

struct ConvParams {
    const uint16_t *qkv, *conv_w;
    const uint16_t *conv_state;   // may be null (zeros)
    const uint8_t *mask;          // may be null
    uint16_t *q, *k, *v;
    int B, T, Hk, Hv, C, K;
    float eps;
};

// Continues a backward scan for the most recent valid steps of row b: nf
// holds `found` positions (newest first), the scan resumes below `cur`.
// Positions older than the first valid token become conv_state codes (< 0,
// -1 = newest stored row).  Warp-collective.
__device__ __forceinline__ void scan_halo(const uint8_t *mask, int b, int T, int cur, int found, int lane,
                                          int (&nf)[kMaxHalo]) {
    while (found < kMaxHalo && cur > 0) {
        const int base = max(cur - 32, 0);
        const int len = cur - base;
        const bool m = lane < len && mask[(size_t)b * T + base + lane] != 0;
        unsigned ball = __ballot_sync(0xffffffffu, m);
        while (ball != 0u && found < kMaxHalo) {
            const int hi = 31 - __clz(ball);
#pragma unroll
            for (int r = 0; r < kMaxHalo; ++r)
                if (r == found) nf[r] = base + hi;
            ++found;
            ball &= ~(1u << hi);
        }
        cur = base;
    }
#pragma unroll
    for (int r = 0; r < kMaxHalo; ++r)
        if (r >= found) nf[r] = -(r - found + 1);
}

// Positions of the kMaxHalo most recent valid steps strictly before `t_end` of
// row b, oldest first.  A code >= 0 is a token index; a code < 0 names
// conv_state row (K-1+code) (-1 = newest stored row).  Warp-collective.
__device__ __forceinline__ void find_halo(const uint8_t *mask, int b, int T, int t_end, int lane,
                                          int (&codes)[kMaxHalo]) {
    int nf[kMaxHalo];   // newest first
    if (mask == nullptr) {
#pragma unroll
        for (int r = 0; r < kMaxHalo; ++r) nf[r] = t_end - 1 - r;
    } else {
        int found = 0;
#pragma unroll
        for (int r = 0; r < kMaxHalo; ++r) nf[r] = 0;
        int cur = t_end;
        while (found < kMaxHalo && cur > 0) {
            const int base = max(cur - 32, 0);
            const int len = cur - base;
            const bool m = lane < len && mask[(size_t)b * T + base + lane] != 0;
            unsigned ball = __ballot_sync(0xffffffffu, m);
            while (ball != 0u && found < kMaxHalo) {
                const int hi = 31 - __clz(ball);
#pragma unroll
                for (int r = 0; r < kMaxHalo; ++r)
                    if (r == found) nf[r] = base + hi;
                ++found;
                ball &= ~(1u << hi);
            }
            cur = base;
        }
        // steps older than the first valid token come from conv_state
#pragma unroll
        for (int r = 0; r < kMaxHalo; ++r)
            if (r >= found) nf[r] = -(r - found + 1);
    }
#pragma unroll
    for (int j = 0; j < kMaxHalo; ++j) codes[j] = nf[kMaxHalo - 1 - j];
}

template <int CPL>
__device__ __forceinline__ void load_bf16(const uint16_t *p, float (&o)[CPL]) {
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
__device__ __forceinline__ void store_bf16(uint16_t *p, const float (&x)[CPL]) {
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

template <int CPL>
__device__ __forceinline__ void store_zero(uint16_t *p) {
    if constexpr (CPL == 4) *reinterpret_cast<uint2 *>(p) = make_uint2(0u, 0u);
    else if constexpr (CPL == 2) *reinterpret_cast<uint32_t *>(p) = 0u;
    else *p = 0;
}

// One head segment of D channels (c0 = first channel) over one token tile.
// kind: 0 = q (rms-norm, scale 1/D), 1 = k (rms-norm, scale 1/sqrt(D)), 2 = v.
template <int D>
__device__ __forceinline__ void conv_segment(const ConvParams &p, int kind, int c0, uint16_t *out_base,
                                             int out_head_stride, int b, int t0, int lane) {
    constexpr int CPL = D / 32;
    const int c = c0 + lane * CPL;
    const int nt = min(kTile, p.T - t0);

    // One mask load for the tile and the 24 steps before it: lanes 0-23 read
    // steps t0-24 .. t0-1 (candidates for the window rows before the tile),
    // lanes 24-31 the tile itself.
    constexpr int kPre = 32 - kTile;
    unsigned valid, prev = 0u;
    if (p.mask != nullptr) {
        const int t = t0 - kPre + lane;
        const bool in = lane < kPre ? t >= 0 : lane - kPre < nt;
        const bool m = in && p.mask[(size_t)b * p.T + t] != 0;
        const unsigned ball = __ballot_sync(0xffffffffu, m);
        valid = ball >> kPre;
        prev = ball & ((1u << kPre) - 1u);
    } else {
        valid = nt >= 32 ? 0xffffffffu : ((1u << nt) - 1u);
    }
    // out element (b, t, head, lane*CPL): out_base already points at (b, 0, head, 0)
    auto out_ptr = [&](int t) { return out_base + (size_t)t * out_head_stride + lane * CPL; };

    if (valid == 0u) {
        for (int i = 0; i < nt; ++i) store_zero<CPL>(out_ptr(t0 + i));
        return;
    }

    // taps, right-aligned to 4 (tap K-1 of the page's weight -> slot 3)
    float w[CPL][4];
#pragma unroll
    for (int i = 0; i < CPL; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int jj = j - (4 - p.K);
            w[i][j] = jj >= 0 ? bf16_to_f32(p.conv_w[(size_t)(c + i) * p.K + jj]) : 0.0f;
        }

    // window of the K-1 valid rows before the tile (zeros for unused slots):
    // the newest valid steps among the 24 already seen, the rest (rarely
    // needed) by scanning further back
    int codes[kMaxHalo];
    if (p.mask == nullptr) {
#pragma unroll
        for (int j = 0; j < kMaxHalo; ++j) codes[j] = t0 - kMaxHalo + j;
    } else {
        int nf[kMaxHalo] = {0, 0, 0};
        int found = 0;
        unsigned pb = prev;
#pragma unroll
        for (int r = 0; r < kMaxHalo; ++r) {
            if (pb != 0u) {
                const int hi = 31 - __clz(pb);
                nf[r] = t0 - kPre + hi;
                pb &= ~(1u << hi);
                found = r + 1;
            }
        }
        if (found < kMaxHalo) scan_halo(p.mask, b, p.T, t0 - kPre, found, lane, nf);
#pragma unroll
        for (int j = 0; j < kMaxHalo; ++j) codes[j] = nf[kMaxHalo - 1 - j];
    }
    float win[kMaxHalo][CPL];
#pragma unroll
    for (int j = 0; j < kMaxHalo; ++j) {
        const int code = codes[j];
        const bool used = j >= kMaxHalo - (p.K - 1);
#pragma unroll
        for (int i = 0; i < CPL; ++i) win[j][i] = 0.0f;
        if (used) {
            if (code >= 0) {
                load_bf16<CPL>(p.qkv + ((size_t)b * p.T + code) * p.C + c, win[j]);
            } else if (p.conv_state != nullptr && p.K - 1 + code >= 0) {
                load_bf16<CPL>(p.conv_state + ((size_t)b * (p.K - 1) + (p.K - 1 + code)) * p.C + c, win[j]);
            }
        }
    }

    // all tile rows in flight at once
    float xr[kTile][CPL];
#pragma unroll
    for (int r = 0; r < kTile; ++r) {
        if (r < nt && ((valid >> r) & 1u)) {
            load_bf16<CPL>(p.qkv + ((size_t)b * p.T + t0 + r) * p.C + c, xr[r]);
        } else {
#pragma unroll
            for (int i = 0; i < CPL; ++i) xr[r][i] = 0.0f;
        }
    }

    const float inv_d = 1.0f / (float)D;
    const float scale = kind == 0 ? inv_d : (kind == 1 ? 1.0f / sqrtf((float)D) : 1.0f);
#pragma unroll
    for (int r = 0; r < kTile; ++r) {
        if (r >= nt) break;
        uint16_t *op = out_ptr(t0 + r);
        if (!((valid >> r) & 1u)) {
            store_zero<CPL>(op);
            continue;
        }
        float x[CPL];
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            float u = w[i][0] * win[0][i];
            u = fmaf(w[i][1], win[1][i], u);
            u = fmaf(w[i][2], win[2][i], u);
            u = fmaf(w[i][3], xr[r][i], u);
            x[i] = silu(u);
            ss = fmaf(x[i], x[i], ss);
        }
        if (kind != 2) {
            ss = warp_sum(ss);
            const float rs = (1.0f / sqrtf(ss * inv_d + p.eps)) * scale;
#pragma unroll
            for (int i = 0; i < CPL; ++i) x[i] *= rs;
        }
        store_bf16<CPL>(op, x);
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            win[0][i] = win[1][i];
            win[1][i] = win[2][i];
            win[2][i] = xr[r][i];
        }
    }
}

template <int DK, int DV>
__global__ void __launch_bounds__(kWarps * 32, 4) conv_update_kernel(const ConvParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.y * kWarps + warp;
    const int nseg = 2 * p.Hk + p.Hv;
    if (seg >= nseg) return;
    const int t0 = blockIdx.x * kTile;
    const int b = blockIdx.z;
    if (seg < p.Hk) {
        uint16_t *ob = p.q + ((size_t)b * p.T * p.Hk + seg) * DK;
        conv_segment<DK>(p, 0, seg * DK, ob, p.Hk * DK, b, t0, lane);
    } else if (seg < 2 * p.Hk) {
        const int hk = seg - p.Hk;
        uint16_t *ob = p.k + ((size_t)b * p.T * p.Hk + hk) * DK;
        conv_segment<DK>(p, 1, seg * DK, ob, p.Hk * DK, b, t0, lane);
    } else {
        const int hv = seg - 2 * p.Hk;
        uint16_t *ob = p.v + ((size_t)b * p.T * p.Hv + hv) * DV;
        conv_segment<DV>(p, 2, 2 * p.Hk * DK + hv * DV, ob, p.Hv * DV, b, t0, lane);
    }
}

// New conv_state = the K-1 newest rows of [conv_state || valid tokens].
__global__ void __launch_bounds__(256) conv_state_kernel(const ConvParams p, uint16_t *conv_state) {
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    int codes[kMaxHalo];
    find_halo(p.mask, b, p.T, p.T, lane, codes);
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= p.C) return;
    const int n = p.K - 1;
    uint16_t vals[kMaxHalo];
#pragma unroll
    for (int j = 0; j < kMaxHalo; ++j) {
        vals[j] = 0;
        if (j < n) {
            const int code = codes[kMaxHalo - n + j];
            if (code >= 0) vals[j] = p.qkv[((size_t)b * p.T + code) * p.C + c];
            else vals[j] = conv_state[((size_t)b * n + (n + code)) * p.C + c];
        }
    }
#pragma unroll
    for (int j = 0; j < kMaxHalo; ++j)
        if (j < n) conv_state[((size_t)b * n + j) * p.C + c] = vals[j];
}

__global__ void __launch_bounds__(256) gating_kernel(const uint16_t *__restrict__ a, const uint16_t *__restrict__ bb,
                                                     const float *__restrict__ A_log,
                                                     const float *__restrict__ dt_bias, float *__restrict__ g,
                                                     float *__restrict__ beta, size_t n, int Hv) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int h = (int)(i % (size_t)Hv);
        const float x = bf16_to_f32(a[i]) + dt_bias[h];
        g[i] = expf(-expf(A_log[h]) * softplus(x));
        beta[i] = sigmoid(bf16_to_f32(bb[i]));
    }
}

template <int DK, int DV>
cudaError_t launch_conv_t(const ConvParams &p, cudaStream_t st) {
    const int nseg = 2 * p.Hk + p.Hv;
    dim3 grid((p.T + kTile - 1) / kTile, (nseg + kWarps - 1) / kWarps, p.B);
    conv_update_kernel<DK, DV><<<grid, kWarps * 32, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv_update(const Sizes &s, const uint16_t *qkv, const uint16_t *conv_w, uint16_t *conv_state,
                               const uint8_t *mask, uint16_t *q, uint16_t *k, uint16_t *v, cudaStream_t st) {
    ConvParams p{qkv, conv_w, conv_state, mask, q, k, v, s.B, s.T, s.Hk, s.Hv, s.C(), s.K, s.eps};
    cudaError_t e = cudaErrorInvalidValue;
#define GDN_CONV_CASE(DK_, DV_) \
    if (s.Dk == DK_ && s.Dv == DV_) e = launch_conv_t<DK_, DV_>(p, st);
    GDN_CONV_CASE(32, 32) GDN_CONV_CASE(32, 64) GDN_CONV_CASE(32, 128)
    GDN_CONV_CASE(64, 32) GDN_CONV_CASE(64, 64) GDN_CONV_CASE(64, 128)
    GDN_CONV_CASE(128, 32) GDN_CONV_CASE(128, 64) GDN_CONV_CASE(128, 128)
#undef GDN_CONV_CASE
    if (e != cudaSuccess) return e;
    if (conv_state != nullptr) {
        dim3 grid((p.C + 255) / 256, p.B);
        conv_state_kernel<<<grid, 256, 0, st>>>(p, conv_state);
        e = cudaGetLastError();
    }
    return e;
}

cudaError_t launch_gating(const Sizes &s, const uint16_t *a, const uint16_t *b, const float *A_log,
                          const float *dt_bias, float *g, float *beta, cudaStream_t st) {
    const size_t n = (size_t)s.B * s.T * s.Hv;
    const int threads = 256;
    size_t blocks = (n + threads - 1) / threads;
    const size_t cap = (size_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    gating_kernel<<<(unsigned)blocks, threads, 0, st>>>(a, b, A_log, dt_bias, g, beta, n, s.Hv);
    return cudaGetLastError();
}

}  // namespace gdn
