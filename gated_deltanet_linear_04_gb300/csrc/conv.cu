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
// tile of 32 consecutive tokens (three 8-warp CTAs resident per SM).  Each
// lane holds D/32 channels.  The taps and the K-1 window rows before the tile
// are loaded once; the tile is walked in sub-tiles of 4 tokens with the next
// sub-tile's rows in flight, keeping the last K-1 *valid* rows in registers
// (as packed bf16), so every qkv element is read once.  The sub-tile loop is
// not unrolled: the unrolled form missed the instruction cache (measured
// 1.2x slower).  The rms-norm is a warp shuffle sum.
//
// Masked steps ("skip" reading): they do not enter the conv window; their q/k/v
// are written as zeros.  The K-1 valid rows preceding a tile are found by a
// warp-ballot scan backwards over the mask (128 steps per iteration through
// wholly masked stretches); missing rows come from conv_state.
// The new conv_state is written by a second, tiny kernel that runs after the
// first on the stream, because tiles anywhere in the row may still read the
// old conv_state.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace gdn {
namespace {

constexpr int kTile = 32;       // tokens per warp tile (its validity bits are one warp ballot)
constexpr int kSub = 4;         // tokens per sub-tile (one sub-tile's rows in flight ahead)
static_assert(kTile == 32, "a tile's validity bits are one 32-lane ballot");
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
        const uint8_t *mrow = mask + (size_t)b * T;
        while (found < kMaxHalo && cur > 0) {
            // 128-step blocks without a valid step (the padding of a short
            // row) are skipped four mask bytes per lane at a time
            if (cur >= 128 && (reinterpret_cast<uintptr_t>(mrow + cur - 128) & 3u) == 0) {
                const uint32_t wv = *reinterpret_cast<const uint32_t *>(mrow + cur - 128 + 4 * lane);
                if (__ballot_sync(0xffffffffu, wv != 0u) == 0u) {
                    cur -= 128;
                    continue;
                }
            }
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

template <int CPL> struct RawRow;
template <> struct RawRow<4> { using type = uint2; };
template <> struct RawRow<2> { using type = uint32_t; };
template <> struct RawRow<1> { using type = uint16_t; };

template <int CPL>
__device__ __forceinline__ typename RawRow<CPL>::type load_raw(const uint16_t *p) {
    return *reinterpret_cast<const typename RawRow<CPL>::type *>(p);
}

template <int CPL>
__device__ __forceinline__ void unpack(const typename RawRow<CPL>::type &r, float (&o)[CPL]) {
    if constexpr (CPL == 4) {
        o[0] = __uint_as_float(r.x << 16);
        o[1] = __uint_as_float(r.x & 0xffff0000u);
        o[2] = __uint_as_float(r.y << 16);
        o[3] = __uint_as_float(r.y & 0xffff0000u);
    } else if constexpr (CPL == 2) {
        o[0] = __uint_as_float(r << 16);
        o[1] = __uint_as_float(r & 0xffff0000u);
    } else {
        o[0] = bf16_to_f32(r);
    }
}

// One head segment of D channels (c0 = first channel) over one tile of kTile
// tokens, walked in sub-tiles of kSub: the taps and the K-1 window rows
// before the tile are loaded once; the next sub-tile's rows are in flight
// while the current one is computed; the window of the last K-1 valid rows
// travels in registers.
// kind: 0 = q (rms-norm, scale 1/D), 1 = k (rms-norm, scale 1/sqrt(D)), 2 = v.
template <int D>
__device__ __forceinline__ void conv_segment(const ConvParams &p, int kind, int c0, uint16_t *out_base,
                                             int out_head_stride, int b, int t0, int lane) {
    constexpr int CPL = D / 32;
    constexpr int NS = kTile / kSub;
    using Raw = typename RawRow<CPL>::type;
    const int c = c0 + lane * CPL;
    const int nt = min(kTile, p.T - t0);

    unsigned valid;   // bit i: step t0 + i is valid
    if (p.mask != nullptr) {
        const bool m = lane < nt && p.mask[(size_t)b * p.T + t0 + lane] != 0;
        valid = __ballot_sync(0xffffffffu, m);
    } else {
        valid = nt >= 32 ? 0xffffffffu : ((1u << nt) - 1u);
    }
    // out element (b, t, head, lane*CPL): out_base already points at (b, 0, head, 0)
    auto out_ptr = [&](int t) { return out_base + (size_t)t * out_head_stride + lane * CPL; };

    if (valid == 0u) {
        for (int i = 0; i < nt; ++i) store_zero<CPL>(out_ptr(t0 + i));
        return;
    }

    // rows of sub-tile s in flight into buffer `slot` (masked or absent rows read nothing)
    Raw buf[2][kSub];
    auto issue = [&](int s, int slot) {
#pragma unroll
        for (int r = 0; r < kSub; ++r) {
            const int tl = s * kSub + r;
            buf[slot][r] = Raw{};
            if (tl < nt && ((valid >> tl) & 1u))
                buf[slot][r] = load_raw<CPL>(p.qkv + ((size_t)b * p.T + t0 + tl) * p.C + c);
        }
    };
    issue(0, 0);

    // taps, right-aligned to 4 (tap K-1 of the page's weight -> slot 3), kept
    // as bf16 bit patterns (exact; unpacked at use)
    uint16_t w[CPL][4];
#pragma unroll
    for (int i = 0; i < CPL; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int jj = j - (4 - p.K);
            w[i][j] = jj >= 0 ? p.conv_w[(size_t)(c + i) * p.K + jj] : (uint16_t)0;
        }

    // window of the K-1 valid rows before the tile (zeros for unused slots),
    // kept as the raw bf16 rows
    int codes[kMaxHalo];
    find_halo(p.mask, b, p.T, t0, lane, codes);
    Raw win[kMaxHalo];
#pragma unroll
    for (int j = 0; j < kMaxHalo; ++j) {
        const int code = codes[j];
        const bool used = j >= kMaxHalo - (p.K - 1);
        win[j] = Raw{};
        if (used) {
            if (code >= 0) {
                win[j] = load_raw<CPL>(p.qkv + ((size_t)b * p.T + code) * p.C + c);
            } else if (p.conv_state != nullptr && p.K - 1 + code >= 0) {
                win[j] = load_raw<CPL>(p.conv_state + ((size_t)b * (p.K - 1) + (p.K - 1 + code)) * p.C + c);
            }
        }
    }

    const float inv_d = 1.0f / (float)D;
    const float scale = kind == 0 ? inv_d : (kind == 1 ? 1.0f / sqrtf((float)D) : 1.0f);
    // one sub-tile from buffer SLOT (a compile-time index, so the rows stay
    // in registers); the sub-tile loop itself is not unrolled, which keeps the
    // code within the instruction cache
    auto sub_tile = [&](auto slot_c, int s) {
        constexpr int SLOT = decltype(slot_c)::value;
#pragma unroll
        for (int r = 0; r < kSub; ++r) {
            const int tl = s * kSub + r;
            if (tl >= nt) break;
            uint16_t *op = out_ptr(t0 + tl);
            if (!((valid >> tl) & 1u)) {
                store_zero<CPL>(op);
                continue;
            }
            float xr[CPL], w0[CPL], w1[CPL], w2[CPL];
            unpack<CPL>(buf[SLOT][r], xr);
            unpack<CPL>(win[0], w0);
            unpack<CPL>(win[1], w1);
            unpack<CPL>(win[2], w2);
            float x[CPL];
            float ss = 0.0f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                float u = bf16_to_f32(w[i][0]) * w0[i];
                u = fmaf(bf16_to_f32(w[i][1]), w1[i], u);
                u = fmaf(bf16_to_f32(w[i][2]), w2[i], u);
                u = fmaf(bf16_to_f32(w[i][3]), xr[i], u);
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
            win[0] = win[1];
            win[1] = win[2];
            win[2] = buf[SLOT][r];
        }
    };
#pragma unroll 1
    for (int s = 0; s < NS && s * kSub < nt; s += 2) {
        if (s + 1 < NS) issue(s + 1, 1);
        sub_tile(std::integral_constant<int, 0>{}, s);
        if (s + 1 >= NS || (s + 1) * kSub >= nt) break;
        if (s + 2 < NS) issue(s + 2, 0);
        sub_tile(std::integral_constant<int, 1>{}, s + 1);
    }
}

template <int DK, int DV>
__global__ void __launch_bounds__(kWarps * 32, 3) conv_update_kernel(const ConvParams p) {
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
