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
// tile of 32 consecutive tokens (three 8-warp CTAs resident per SM).  The
// tile's rows arrive in shared memory by one TMA copy (a [32 x D] box of a
// 3-D tensor map over qkv, clipped at the row's T), issued first, so every
// resident warp has its whole tile in flight while it loads the taps and the
// K-1 window rows before the tile.  Each lane then holds D/32 channels; the
// window of the last K-1 *valid* rows travels in registers.  The arithmetic
// runs on channel pairs with the packed two-wide f32 instructions of sm_100,
// and the q/k rms-norm sums four tokens per warp reduction (six shuffles).
//
// Masked steps ("skip" reading): they do not enter the conv window; their q/k/v
// are written as zeros.  A tile without a valid step copies nothing.  The K-1
// valid rows preceding a tile are found by a warp-ballot scan backwards over
// the mask (128 steps per iteration through wholly masked stretches); missing
// rows come from conv_state.
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
    unsigned *err;
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

// Channel pairs of one lane: CPL channels as NP float2 (CPL = 1 uses the
// low half only).  The arithmetic on them is the packed two-wide f32 form of
// sm_100 (fma.rn.f32x2 and friends), each half rounded exactly like the
// scalar instruction, so a pair costs one instruction where two scalars did.
template <int CPL> struct Pairs { static constexpr int NP = CPL >= 2 ? CPL / 2 : 1; float2 v[NP]; };

template <int CPL>
__device__ __forceinline__ Pairs<CPL> unpack_pairs(const typename RawRow<CPL>::type &r) {
    Pairs<CPL> o;
    if constexpr (CPL == 4) {
        o.v[0] = make_float2(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u));
        o.v[1] = make_float2(__uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
    } else if constexpr (CPL == 2) {
        o.v[0] = make_float2(__uint_as_float(r << 16), __uint_as_float(r & 0xffff0000u));
    } else {
        o.v[0] = make_float2(bf16_to_f32(r), 0.0f);
    }
    return o;
}

// Two bf16 (RNE) in one 32-bit word, low half first.
__device__ __forceinline__ uint32_t pack_bf16x2(float2 x) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x.x, x.y);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int CPL>
__device__ __forceinline__ void store_pairs(uint16_t *p, const Pairs<CPL> &x) {
    if constexpr (CPL == 4) *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(x.v[0]), pack_bf16x2(x.v[1]));
    else if constexpr (CPL == 2) *reinterpret_cast<uint32_t *>(p) = pack_bf16x2(x.v[0]);
    else *p = f32_to_bf16(x.v[0].x);
}

// silu(u) = u * sigmoid(u) on a pair, with the hardware base-2 exponential
// and reciprocal (the same operations as the scalar silu of common.cuh)
__device__ __forceinline__ float2 silu2(float2 u) {
    const float2 t = __fmul2_rn(u, make_float2(-1.4426950408889634f, -1.4426950408889634f));
    float e0, e1;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t.x));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t.y));
    const float2 d = __fadd2_rn(make_float2(e0, e1), make_float2(1.0f, 1.0f));
    return __fmul2_rn(u, make_float2(rcp_fast(d.x), rcp_fast(d.y)));
}

// Warp sums of four per-lane values s[0..3] (one per token of a sub-tile) in
// six shuffles: two halving exchanges hand each lane half, then a quarter,
// of the tokens, and three more rounds finish the sum.  The result is the
// total of token ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1).
__device__ __forceinline__ float warp_sum4(const float (&s)[4], int lane) {
    const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
    float a0 = h16 ? s[2] : s[0], a1 = h16 ? s[3] : s[1];
    const float b0 = h16 ? s[0] : s[2], b1 = h16 ? s[1] : s[3];
    a0 += __shfl_xor_sync(0xffffffffu, b0, 16);
    a1 += __shfl_xor_sync(0xffffffffu, b1, 16);
    float k = h8 ? a1 : a0;
    const float o = h8 ? a0 : a1;
    k += __shfl_xor_sync(0xffffffffu, o, 8);
    k += __shfl_xor_sync(0xffffffffu, k, 4);
    k += __shfl_xor_sync(0xffffffffu, k, 2);
    k += __shfl_xor_sync(0xffffffffu, k, 1);
    return k;
}

// One head segment of D channels (c0 = first channel) over one tile of kTile
// tokens, walked in sub-tiles of kSub: the taps and the K-1 window rows
// before the tile are loaded once; the next sub-tile's rows are in flight
// while the current one is computed; the window of the last K-1 valid rows
// travels in registers (as f32 pairs).  A sub-tile is computed in two
// phases: conv + SiLU of its (up to) four tokens with their sums of squares,
// then one four-token warp reduction for the q/k norm, then the scaled
// stores.
// kind: 0 = q (rms-norm, scale 1/D), 1 = k (rms-norm, scale 1/sqrt(D)), 2 = v.
template <int D>
__device__ __forceinline__ void conv_segment(const ConvParams &p, const CUtensorMap *tm, uint8_t *tile,
                                             uint64_t *bar, int kind, int c0, uint16_t *out_base,
                                             int out_head_stride, int b, int t0, int lane) {
    constexpr int CPL = D / 32;
    constexpr int NP = Pairs<CPL>::NP;
    constexpr int NS = kTile / kSub;
    static_assert(kSub == 4, "the norm reduction sums four tokens at once");
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

    // the tile's rows [32][D] by one TMA copy (rows past T read as zeros)
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_expect_tx(bar, kTile * D * 2);
        tma_load_3d(tile, tm, c0, t0, b, bar);
    }
    __syncwarp();   // the barrier's initialisation is seen by every lane before it waits

    // taps, right-aligned to 4 (tap K-1 of the page's weight -> slot 3), as
    // f32 pairs (bf16 values, exact)
    float2 tap[4][NP];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int jj = j - (4 - p.K);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            float lo = 0.0f, hi = 0.0f;
            if (jj >= 0) {
                lo = bf16_to_f32(p.conv_w[(size_t)(c + 2 * i) * p.K + jj]);
                if (CPL >= 2) hi = bf16_to_f32(p.conv_w[(size_t)(c + 2 * i + 1) * p.K + jj]);
            }
            tap[j][i] = make_float2(lo, hi);
        }
    }

    // window of the K-1 valid rows before the tile (zeros for unused slots)
    int codes[kMaxHalo];
    find_halo(p.mask, b, p.T, t0, lane, codes);
    Pairs<CPL> win[kMaxHalo];
#pragma unroll
    for (int j = 0; j < kMaxHalo; ++j) {
        const int code = codes[j];
        const bool used = j >= kMaxHalo - (p.K - 1);
        Raw r = Raw{};
        if (used) {
            if (code >= 0) {
                r = load_raw<CPL>(p.qkv + ((size_t)b * p.T + code) * p.C + c);
            } else if (p.conv_state != nullptr && p.K - 1 + code >= 0) {
                r = load_raw<CPL>(p.conv_state + ((size_t)b * (p.K - 1) + (p.K - 1 + code)) * p.C + c);
            }
        }
        win[j] = unpack_pairs<CPL>(r);
    }

    // every lane waits for the copy (bounded; on expiry the error word is set
    // and the tile is left unwritten)
    if (!mbar_wait(bar, 0, p.err)) return;
    const uint16_t *rows = reinterpret_cast<const uint16_t *>(tile) + lane * CPL;

    const float inv_d = 1.0f / (float)D;
    const float scale = kind == 0 ? inv_d : (kind == 1 ? 1.0f / sqrtf((float)D) : 1.0f);
    // sub-tiles of four tokens: conv + SiLU of each valid token with its sum
    // of squares, one four-token warp reduction for the q/k norm, the stores;
    // the sub-tile loop is not unrolled, which keeps the code within the
    // instruction cache
    // conv + SiLU of one token from its K window rows (oldest first), with
    // its sum of squares
    auto conv_token = [&](const Pairs<CPL> &r0, const Pairs<CPL> &r1, const Pairs<CPL> &r2, const Pairs<CPL> &r3,
                          Pairs<CPL> &x, float &ss) {
        float2 sq = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            float2 u = __fmul2_rn(tap[0][i], r0.v[i]);
            u = __ffma2_rn(tap[1][i], r1.v[i], u);
            u = __ffma2_rn(tap[2][i], r2.v[i], u);
            u = __ffma2_rn(tap[3][i], r3.v[i], u);
            x.v[i] = silu2(u);
            sq = __ffma2_rn(x.v[i], x.v[i], sq);
        }
        ss = CPL >= 2 ? sq.x + sq.y : sq.x;
    };
#pragma unroll 1
    for (int s = 0; s < NS && s * kSub < nt; ++s) {
        Pairs<CPL> x[kSub];
        float ss[kSub];
        if (((valid >> (s * kSub)) & 0xFu) == 0xFu) {
            // four valid tokens: the window rolls by static register indices
            Pairs<CPL> xr[kSub];
#pragma unroll
            for (int r = 0; r < kSub; ++r) xr[r] = unpack_pairs<CPL>(load_raw<CPL>(rows + (s * kSub + r) * D));
            conv_token(win[0], win[1], win[2], xr[0], x[0], ss[0]);
            conv_token(win[1], win[2], xr[0], xr[1], x[1], ss[1]);
            conv_token(win[2], xr[0], xr[1], xr[2], x[2], ss[2]);
            conv_token(xr[0], xr[1], xr[2], xr[3], x[3], ss[3]);
            win[0] = xr[1];
            win[1] = xr[2];
            win[2] = xr[3];
        } else {
            // masked steps (or the tile's end) inside: token by token, only
            // valid tokens entering the window
#pragma unroll
            for (int r = 0; r < kSub; ++r) {
                const int tl = s * kSub + r;
                ss[r] = 0.0f;
#pragma unroll
                for (int i = 0; i < NP; ++i) x[r].v[i] = make_float2(0.0f, 0.0f);
                if (tl < nt && ((valid >> tl) & 1u)) {
                    const Pairs<CPL> xr = unpack_pairs<CPL>(load_raw<CPL>(rows + tl * D));
                    conv_token(win[0], win[1], win[2], xr, x[r], ss[r]);
                    win[0] = win[1];
                    win[1] = win[2];
                    win[2] = xr;
                }
            }
        }
        if (kind != 2) {
            // each lane normalises one token; the four factors are then
            // broadcast from lanes 0, 8, 16 and 24
            const float tot = warp_sum4(ss, lane);
            const float rs_mine = rsqrtf(tot * inv_d + p.eps) * scale;
#pragma unroll
            for (int r = 0; r < kSub; ++r) {
                const float rs = __shfl_sync(0xffffffffu, rs_mine, ((r >> 1) << 4) | ((r & 1) << 3));
#pragma unroll
                for (int i = 0; i < NP; ++i) x[r].v[i] = __fmul2_rn(x[r].v[i], make_float2(rs, rs));
            }
        }
#pragma unroll
        for (int r = 0; r < kSub; ++r) {
            const int tl = s * kSub + r;
            if (tl < nt) store_pairs<CPL>(out_ptr(t0 + tl), x[r]);   // masked steps: zeros
        }
    }
}

// Shared memory of a CTA: one [kTile x max(DK, DV)] bf16 tile per warp, from
// a 128-byte aligned base (the TMA destination alignment).
template <int DK, int DV>
constexpr uint32_t conv_smem_bytes() {
    return (uint32_t)kWarps * kTile * (DK > DV ? DK : DV) * 2 + 128;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kWarps * 32, 3) conv_update_kernel(const __grid_constant__ CUtensorMap tm_qk,
                                                                     const __grid_constant__ CUtensorMap tm_v,
                                                                     const ConvParams p) {
    extern __shared__ __align__(128) uint8_t conv_smem_raw[];
    __shared__ __align__(8) uint64_t bars[kWarps];
    uint8_t *conv_smem = conv_smem_raw + (((smem_u32(conv_smem_raw) + 127u) & ~127u) - smem_u32(conv_smem_raw));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.y * kWarps + warp;
    const int nseg = 2 * p.Hk + p.Hv;
    if (seg >= nseg) return;
    const int t0 = blockIdx.x * kTile;
    const int b = blockIdx.z;
    uint8_t *tile = conv_smem + (size_t)warp * kTile * (DK > DV ? DK : DV) * 2;
    if (seg < p.Hk) {
        uint16_t *ob = p.q + ((size_t)b * p.T * p.Hk + seg) * DK;
        conv_segment<DK>(p, &tm_qk, tile, &bars[warp], 0, seg * DK, ob, p.Hk * DK, b, t0, lane);
    } else if (seg < 2 * p.Hk) {
        const int hk = seg - p.Hk;
        uint16_t *ob = p.k + ((size_t)b * p.T * p.Hk + hk) * DK;
        conv_segment<DK>(p, &tm_qk, tile, &bars[warp], 1, seg * DK, ob, p.Hk * DK, b, t0, lane);
    } else {
        const int hv = seg - 2 * p.Hk;
        uint16_t *ob = p.v + ((size_t)b * p.T * p.Hv + hv) * DV;
        conv_segment<DV>(p, &tm_v, tile, &bars[warp], 2, 2 * p.Hk * DK + hv * DV, ob, p.Hv * DV, b, t0, lane);
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

// Each thread steps its head index by the grid stride modulo Hv instead of
// dividing every element's index (a 64-bit remainder per element was a large
// part of this kernel's instructions); with SMEM (Hv up to kGateSmemHeads)
// the per-head constants exp(A_log) and dt_bias sit in shared memory.  The
// arithmetic per element is the same either way.
constexpr int kGateSmemHeads = 2048;
template <bool SMEM>
__global__ void __launch_bounds__(256) gating_kernel(const uint16_t *__restrict__ a, const uint16_t *__restrict__ bb,
                                                     const float *__restrict__ A_log,
                                                     const float *__restrict__ dt_bias, float *__restrict__ g,
                                                     float *__restrict__ beta, size_t n, int Hv) {
    __shared__ float gate_consts[SMEM ? 2 * kGateSmemHeads : 1];   // [Hv] exp(A_log), [Hv] dt_bias
    if constexpr (SMEM) {
        for (int h = threadIdx.x; h < Hv; h += blockDim.x) {
            gate_consts[h] = expf(A_log[h]);
            gate_consts[kGateSmemHeads + h] = dt_bias[h];
        }
        __syncthreads();
    }
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const int hstep = (int)(stride % (size_t)Hv);
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    int h = (int)(i % (size_t)Hv);
    for (; i < n; i += stride) {
        const float ea = SMEM ? gate_consts[h] : expf(A_log[h]);
        const float x = bf16_to_f32(a[i]) + (SMEM ? gate_consts[kGateSmemHeads + h] : dt_bias[h]);
        g[i] = expf(-ea * softplus(x));
        beta[i] = sigmoid(bf16_to_f32(bb[i]));
        h += hstep;
        if (h >= Hv) h -= Hv;
    }
}

template <int DK, int DV>
cudaError_t launch_conv_t(const ConvParams &p, cudaStream_t st) {
    // 3-D maps over qkv [B][T][C] with a [32 tokens x D channels] box (the
    // box is clipped at each row's T, so a tile never reads the next row)
    CUtensorMap tqk, tv;
    if (!encode_tmap_3d(&tqk, p.qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.B, (uint64_t)p.T,
                        (uint64_t)p.C, kTile, DK) ||
        !encode_tmap_3d(&tv, p.qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.B, (uint64_t)p.T,
                        (uint64_t)p.C, kTile, DV))
        return cudaErrorInvalidValue;
    static unsigned long long attr_done = 0;   // per instantiation, one bit per device
    cudaError_t e = set_max_smem(attr_done, conv_update_kernel<DK, DV>, conv_smem_bytes<DK, DV>());
    if (e != cudaSuccess) return e;
    const int nseg = 2 * p.Hk + p.Hv;
    dim3 grid((p.T + kTile - 1) / kTile, (nseg + kWarps - 1) / kWarps, p.B);
    conv_update_kernel<DK, DV><<<grid, kWarps * 32, conv_smem_bytes<DK, DV>(), st>>>(tqk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv_update(const Sizes &s, const uint16_t *qkv, const uint16_t *conv_w, uint16_t *conv_state,
                               const uint8_t *mask, uint16_t *q, uint16_t *k, uint16_t *v, unsigned *err,
                               cudaStream_t st) {
    ConvParams p{qkv, conv_w, conv_state, mask, q, k, v, err, s.B, s.T, s.Hk, s.Hv, s.C(), s.K, s.eps};
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
    if (blocks == 0) return cudaSuccess;
    if (s.Hv <= kGateSmemHeads)
        gating_kernel<true><<<(unsigned)blocks, threads, 0, st>>>(a, b, A_log, dt_bias, g, beta, n, s.Hv);
    else
        gating_kernel<false><<<(unsigned)blocks, threads, 0, st>>>(a, b, A_log, dt_bias, g, beta, n, s.Hv);
    return cudaGetLastError();
}

}  // namespace gdn
