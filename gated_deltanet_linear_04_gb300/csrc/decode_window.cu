// Multi-token decode window (speculative verify / accepted-prefix commit):
// T <= 8 new tokens per row run through conv window + conv + SiLU + q/k norm,
// the gates and the recurrence in one kernel that streams the f32 state once.
// y is produced for all T tokens; conv_state and the state are advanced by
// exactly keep[b] leading tokens.
//
// Definitions: "mlx-bun 0.4.0 -> 1.0.0, package/src/model/qwen3-delta.ts",
// gated_delta_step (per-step update) and SsmSpecRound / specRoundRollback (a
// verify window over S tokens whose first `keep` tokens are kept, the state
// after them being the same arithmetic prefix); "mlex 0.1.2,
// src/models/gated_delta.rs", GatedDeltaNet::forward (conv window, conv1d +
// silu, q/k normalisation, beta, g).
//
// Layout of the single-token kernel: a cluster per (b, hk) group of the G
// v-heads x SN row slices (here SN = 1, a whole head per CTA, unless the
// heads are too few to fill the GPU), each CTA bulk-copies its R x Dk state
// slice into shared memory while it computes the conv/norm/gates of the T
// tokens.  A
// CTA's life is a chain (inputs -> conv -> norm -> rows -> stores) with the
// state copy hidden under its first links, and with several CTAs per SM the
// links also compete for issue slots, so the chain is kept short: the conv
// windows and taps are loaded at entry (the last warp computes the gates
// while its loads are in flight), the new conv_state is taken from the window
// already in registers, the token loops run branch-free to a compile-time
// bound (4 or 8) over zero-padded tokens, and the q/k normalisation factor
// is formed once per (token, q or k).  Eight lanes walk a row through all T
// tokens with the row in registers: S_{t-1} k, the update, then y = S_t q
// (each lane group carries two rows at once and a warp eight, so a row's dot
// products are 3-level shuffle sums; lane l holds the row's 16-byte
// column groups l, l + 8, ..., which keeps each quarter-warp's shared-memory
// accesses on distinct banks); after token keep-1 the row is written back to
// shared memory, so the slice stored at the end is the state after the kept
// prefix (nothing is stored when keep is 0).
#include "common.cuh"
#include "internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunkRows = 32;
constexpr int kMaxRows = 128;
constexpr int kMaxT = 8;

struct WindowParams {
    const uint16_t *qkv, *conv_w;
    uint16_t *conv_state;
    const uint16_t *a, *b;
    const float *A_log, *dt_bias;
    float *state;
    const int32_t *keep;
    uint16_t *y;
    unsigned *err;
    int B, T, Hk, Hv, Dv, C, K, SN;
    float eps;
};

// The conv window of channel c: x[0 .. K-1) = the stored rows (oldest
// first), x[K-1 + t] = token t (zero past T), and its K taps, as f32 (bf16
// widened exactly, so the top 16 bits are the bf16 bit pattern).
template <int K, int TM>
struct ConvWindow {
    float x[K - 1 + TM];
    float w[K];

    // the taps (constant across calls: read before waiting on the previous grid)
    __device__ __forceinline__ void load_taps(const WindowParams &p, int c) {
#pragma unroll
        for (int j = 0; j < K; ++j) w[j] = bf16_to_f32(p.conv_w[(size_t)c * K + j]);
    }
    __device__ __forceinline__ void load(const WindowParams &p, int b, int c) {
        constexpr int n = K - 1;
        const uint16_t *cs = p.conv_state + (size_t)b * n * p.C + c;
#pragma unroll
        for (int j = 0; j < n; ++j) x[j] = bf16_to_f32(cs[(size_t)j * p.C]);
#pragma unroll
        for (int t = 0; t < TM; ++t) x[n + t] = t < p.T ? bf16_to_f32(p.qkv[((size_t)b * p.T + t) * p.C + c]) : 0.0f;
    }

    // SiLU(conv) of tokens t < TM: taps j = 0 .. K-1 read x[t + j] (the
    // token's own value on tap K-1).
    __device__ __forceinline__ void conv_silu(float (&out)[TM]) const {
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            float u = 0.0f;
#pragma unroll
            for (int j = 0; j < K; ++j) u = fmaf(w[j], x[t + j], u);
            out[t] = silu(u);
        }
    }

    // conv_state rows after the first `keep` (0 .. TM) tokens: row j is
    // window entry keep + j, reached by shifting the rows one entry per kept
    // token (constant indices only, so the window stays in registers).
    __device__ __forceinline__ void new_conv_rows(int keep, uint16_t (&rows)[K - 1]) const {
        float r[K - 1];
#pragma unroll
        for (int j = 0; j < K - 1; ++j) r[j] = x[j];
#pragma unroll
        for (int s = 0; s < TM; ++s)
#pragma unroll
            for (int j = 0; j < K - 1; ++j) r[j] = s < keep ? x[s + 1 + j] : r[j];
#pragma unroll
        for (int j = 0; j < K - 1; ++j) rows[j] = (uint16_t)(__float_as_uint(r[j]) >> 16);
    }
};

template <int K>
__device__ __forceinline__ void store_conv_rows(const WindowParams &p, int b, int c, const uint16_t (&rows)[K - 1]) {
    uint16_t *cs = p.conv_state + (size_t)b * (K - 1) * p.C + c;
#pragma unroll
    for (int j = 0; j < K - 1; ++j) cs[(size_t)j * p.C] = rows[j];
}

// Three CTAs per SM (80 registers, no spills) for loops to at most 6
// tokens, where a CTA holds all 128 rows of a head (64 KiB of state: room for
// three in shared memory anyway); four (64 registers) for loops to 8, which
// take half a head per CTA.
template <int DK, int K, int TM>
__global__ void __launch_bounds__(kThreads, TM == 8 ? 4 : 3) window_kernel(const WindowParams p) {
    constexpr int LPR = 8;             // lanes per row
    constexpr int RPP = 32 / LPR;      // rows per warp pass
    constexpr int NG = DK / 4 / LPR;   // 16-byte column groups per lane
    constexpr int NW = DK / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.Hv / p.Hk;
    const int R = p.Dv / p.SN;
    const int rank = blockIdx.x;
    const int hv_local = rank / p.SN, slice = rank % p.SN;
    const int hk = blockIdx.y, b = blockIdx.z;
    const int hv = hk * G + hv_local;
    const int r0 = slice * R;
    const int T = p.T;
    grid_dep_launch();

    // before the wait only the constant taps; every other input (state,
    // conv_state, qkv, gates, keep) may be written by the previous grid
    const bool has_qk = tid < 2 * DK;
    const int c_qk = tid < DK ? hk * DK + tid : p.Hk * DK + hk * DK + (tid - DK);
    const bool has_v = tid < R;
    const int c_v = 2 * p.Hk * DK + hv * p.Dv + r0 + tid;
    ConvWindow<K, TM> wqk, wv;
    if (has_qk) wqk.load_taps(p, c_qk);
    if (has_v) wv.load_taps(p, c_v);
    grid_dep_wait();
    int keep = p.keep == nullptr ? T : p.keep[b];
    keep = keep < 0 ? 0 : (keep > T ? T : keep);

    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *S = reinterpret_cast<float *>(smem_raw);
    __shared__ __align__(16) float q_s[TM][DK];
    __shared__ __align__(16) float k_s[TM][DK];
    __shared__ float v_s[TM][kMaxRows];
    __shared__ float y_s[TM][kMaxRows];
    __shared__ float red[TM][kWarps];
    __shared__ float gb_s[TM][2];                  // g, beta per token
    __shared__ float fac_s[TM][2];                 // q and k normalisation factor per token
    __shared__ uint16_t qk_rows_s[K - 1][2 * DK];  // new q/k conv_state rows, stored by rank 0 at the end
    __shared__ __align__(8) uint64_t bars[kMaxRows / kChunkRows];

    const int rc = min(R, kChunkRows);
    const int nch = R / rc;
    const uint32_t chunk_bytes = (uint32_t)rc * DK * 4;
    float *gstate = p.state + (((size_t)b * p.Hv + hv) * p.Dv + r0) * DK;

    if (tid == 0) {
        for (int ch = 0; ch < nch; ++ch) mbar_init(&bars[ch], 1);
        fence_mbar_init();
        for (int ch = 0; ch < nch; ++ch) {
            mbar_expect_tx(&bars[ch], chunk_bytes);
            bulk_load(S + (size_t)ch * rc * DK, gstate + (size_t)ch * rc * DK, chunk_bytes, &bars[ch]);
        }
    }

    // ---- every input load first: the q/k and v conv windows
    if (has_qk) wqk.load(p, b, c_qk);
    if (has_v) wv.load(p, b, c_v);
    // the gates, on the last warp while its conv window is in flight
    if (warp == kWarps - 1 && lane < T) {
        const size_t gi = ((size_t)b * T + lane) * p.Hv + hv;
        const float x = bf16_to_f32(p.a[gi]) + p.dt_bias[hv];
        gb_s[lane][0] = expf(-expf(p.A_log[hv]) * softplus(x));
        gb_s[lane][1] = sigmoid(bf16_to_f32(p.b[gi]));
    }

    // ---- conv + SiLU (tokens past T are zero throughout, so every token
    // loop below runs to TM without a branch); the v channels' conv_state is
    // this CTA's alone and is rewritten at once, the q/k channels' (read by
    // the whole cluster) by rank 0 at the end
    float xqk[TM];
#pragma unroll
    for (int t = 0; t < TM; ++t) xqk[t] = 0.0f;
    if (has_qk) {
        wqk.conv_silu(xqk);
        if (keep > 0) {
            uint16_t rows[K - 1];
            wqk.new_conv_rows(keep, rows);
#pragma unroll
            for (int j = 0; j < K - 1; ++j) qk_rows_s[j][tid] = rows[j];
        }
    }
#pragma unroll
    for (int t = 0; t < TM; ++t)
        if (t >= T) xqk[t] = 0.0f;
    if (has_v) {
        float xv[TM];
        wv.conv_silu(xv);
#pragma unroll
        for (int t = 0; t < TM; ++t) v_s[t][tid] = t < T ? round_bf16(xv[t]) : 0.0f;
        if (keep > 0) {
            uint16_t rows[K - 1];
            wv.new_conv_rows(keep, rows);
            store_conv_rows<K>(p, b, c_v, rows);
        }
    }
    cluster_arrive_relaxed();      // the shared q/k conv_state has been read

    // ---- q/k normalisation: sums of squares 32 channels per warp, one
    // factor per (token, q or k), then each channel scaled and rounded
#pragma unroll
    for (int t = 0; t < TM; ++t) {
        const float ss = warp_sum(xqk[t] * xqk[t]);
        if (lane == 0) red[t][warp] = ss;
    }
    __syncthreads();
    if (tid < 2 * TM) {
        const int t = tid >> 1, part = tid & 1;
        const float inv_d = 1.0f / (float)DK;
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) tot += red[t][part * NW + w];
        fac_s[t][part] = (1.0f / sqrtf(tot * inv_d + p.eps)) * (part ? 1.0f / sqrtf((float)DK) : inv_d);
    }
    __syncthreads();
    if (has_qk) {
        const int part = tid >= DK;
        float *dst = part ? &k_s[0][tid - DK] : &q_s[0][tid];
#pragma unroll
        for (int t = 0; t < TM; ++t) dst[t * DK] = round_bf16(xqk[t] * fac_s[t][part]);
    }
    __syncthreads();

    // ---- rows through the window: each group of eight lanes carries two
    // rows (RPP apart), two independent chains sharing the k / q loads
    const int sub = lane / LPR, cl = lane % LPR;
    bool ok_all = true;
    for (int p0 = warp * 2 * RPP; p0 < R; p0 += kWarps * 2 * RPP) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[p0 / rc], 0, p.err));
        ok_all = ok_all && ok;
        if (!ok) continue;
        const int ra = p0 + sub, rb = ra + RPP;
        float4 *spa = reinterpret_cast<float4 *>(S + (size_t)ra * DK);
        float4 *spb = reinterpret_cast<float4 *>(S + (size_t)rb * DK);
        float4 sa[NG], sb[NG];
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            sa[j] = spa[j * LPR + cl];
            sb[j] = spb[j * LPR + cl];
        }
        for (int t = 0; t < T; ++t) {
            const float4 *k4 = reinterpret_cast<const float4 *>(k_s[t]);
            const float4 *q4 = reinterpret_cast<const float4 *>(q_s[t]);
            const float g = gb_s[t][0], beta = gb_s[t][1];
            // S_{t-1} k, then S_t = g S_{t-1} + delta k^T, then y = S_t q, on
            // column pairs with the packed two-wide f32 instructions (each
            // half rounds like the scalar one; the pair's halves are the two
            // partial sums)
            float2 pa = make_float2(0.0f, 0.0f), pb = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < NG; ++j) {
                const float4 kk = k4[j * LPR + cl];
                pa = __ffma2_rn(make_float2(sa[j].x, sa[j].y), make_float2(kk.x, kk.y), pa);
                pa = __ffma2_rn(make_float2(sa[j].z, sa[j].w), make_float2(kk.z, kk.w), pa);
                pb = __ffma2_rn(make_float2(sb[j].x, sb[j].y), make_float2(kk.x, kk.y), pb);
                pb = __ffma2_rn(make_float2(sb[j].z, sb[j].w), make_float2(kk.z, kk.w), pb);
            }
            float dka = pa.x + pa.y, dkb = pb.x + pb.y;
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) {
                dka += __shfl_xor_sync(0xffffffffu, dka, o);
                dkb += __shfl_xor_sync(0xffffffffu, dkb, o);
            }
            const float da = beta * (v_s[t][ra] - g * dka);
            const float db = beta * (v_s[t][rb] - g * dkb);
            const float2 g2 = make_float2(g, g), da2 = make_float2(da, da), db2 = make_float2(db, db);
            pa = pb = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < NG; ++j) {
                const float4 kk = k4[j * LPR + cl];
                const float4 qq = q4[j * LPR + cl];
                float2 lo = __ffma2_rn(da2, make_float2(kk.x, kk.y), __fmul2_rn(g2, make_float2(sa[j].x, sa[j].y)));
                float2 hi = __ffma2_rn(da2, make_float2(kk.z, kk.w), __fmul2_rn(g2, make_float2(sa[j].z, sa[j].w)));
                sa[j] = make_float4(lo.x, lo.y, hi.x, hi.y);
                pa = __ffma2_rn(lo, make_float2(qq.x, qq.y), pa);
                pa = __ffma2_rn(hi, make_float2(qq.z, qq.w), pa);
                lo = __ffma2_rn(db2, make_float2(kk.x, kk.y), __fmul2_rn(g2, make_float2(sb[j].x, sb[j].y)));
                hi = __ffma2_rn(db2, make_float2(kk.z, kk.w), __fmul2_rn(g2, make_float2(sb[j].z, sb[j].w)));
                sb[j] = make_float4(lo.x, lo.y, hi.x, hi.y);
                pb = __ffma2_rn(lo, make_float2(qq.x, qq.y), pb);
                pb = __ffma2_rn(hi, make_float2(qq.z, qq.w), pb);
            }
            float dqa = pa.x + pa.y, dqb = pb.x + pb.y;
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) {
                dqa += __shfl_xor_sync(0xffffffffu, dqa, o);
                dqb += __shfl_xor_sync(0xffffffffu, dqb, o);
            }
            if (cl == 0) {
                y_s[t][ra] = dqa;
                y_s[t][rb] = dqb;
            }
            if (t == keep - 1) {              // the state after the kept prefix
#pragma unroll
                for (int j = 0; j < NG; ++j) {
                    spa[j * LPR + cl] = sa[j];
                    spb[j * LPR + cl] = sb[j];
                }
            }
        }
    }
    fence_proxy_async_smem();
    ok_all = __syncthreads_and(ok_all) != 0;
    if (ok_all && keep > 0 && tid == 0) {
        bulk_store(gstate, S, (uint32_t)R * DK * 4);
        bulk_commit();
    }
    if (ok_all) {
        // bf16 pairs, token and row by shift and mask: R is a power of two
        // (Dv / SN with Dv in {32, 64, 128}); a division by the runtime R
        // here measured 6 % of the 4-token window
        const int lr = 31 - __clz(R >> 1);
        for (int i = tid; i < T * (R >> 1); i += kThreads) {
            const int t = i >> lr, r = (i & ((R >> 1) - 1)) * 2;
            const __nv_bfloat162 h = __floats2bfloat162_rn(y_s[t][r], y_s[t][r + 1]);
            *reinterpret_cast<__nv_bfloat162 *>(p.y + (((size_t)b * T + t) * p.Hv + hv) * p.Dv + r0 + r) = h;
        }
    }

    // ---- q/k conv_state after the kept prefix: rank 0 writes it once every
    // CTA of the cluster has read it
    cluster_wait_acquire();
    if (keep > 0 && has_qk && rank == 0) {
        uint16_t rows[K - 1];
#pragma unroll
        for (int j = 0; j < K - 1; ++j) rows[j] = qk_rows_s[j][tid];
        store_conv_rows<K>(p, b, c_qk, rows);
    }
    if (tid == 0) bulk_wait_read();   // the slice has been read out of shared memory
}

template <int DK, int K, int TM>
cudaError_t launch_t(const WindowParams &p, cudaStream_t st) {
    const int G = p.Hv / p.Hk;
    const int R = p.Dv / p.SN;
    static unsigned long long attr_done = 0;   // per instantiation, one bit per device
    cudaError_t ae = once_per_device(attr_done, [] {
        cudaError_t e = cudaFuncSetAttribute(window_kernel<DK, K, TM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(kMaxRows * DK * sizeof(float)));
        if (e != cudaSuccess) return e;
        return cudaFuncSetAttribute(window_kernel<DK, K, TM>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    });
    if (ae != cudaSuccess) return ae;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G * p.SN, p.Hk, p.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)R * DK * sizeof(float);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G * p.SN;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // programmatic launch (the next grid scheduled while this one drains)
    // only for grids larger than one resident wave, as for the decode step,
    // and not for loops to 6 tokens (it measured 1-2 % slower there, 1-2 %
    // faster for 1, 3, 4 and 7 tokens)
    const long ctas = (long)cfg.gridDim.x * cfg.gridDim.y * cfg.gridDim.z;
    cfg.numAttrs = (TM != 6 && ctas > (TM == 8 ? 4L : 3L) * num_sms()) ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, window_kernel<DK, K, TM>, p);
}

// Token loops run to the smallest of 2, 4, 6, 8 that holds the window (work
// on padded tokens is not free: a 4-token window with loops to 8 measured
// 172 vs 118 us at B=128).
template <int DK, int K>
cudaError_t launch_tm(const WindowParams &p, cudaStream_t st) {
    if (p.T <= 2) return launch_t<DK, K, 2>(p, st);
    if (p.T <= 4) return launch_t<DK, K, 4>(p, st);
    if (p.T <= 6) return launch_t<DK, K, 6>(p, st);
    return launch_t<DK, K, kMaxT>(p, st);
}

}  // namespace

cudaError_t launch_decode_window(const Sizes &s, const uint16_t *qkv, const uint16_t *conv_w, uint16_t *conv_state,
                                 const uint16_t *a, const uint16_t *b, const float *A_log, const float *dt_bias,
                                 float *state, const int32_t *keep, uint16_t *y, unsigned *err, cudaStream_t st) {
    if (s.T < 1 || s.T > kMaxT) return cudaErrorNotSupported;
    // Up to 6 tokens a CTA takes all Dv rows of its head unless the heads are
    // too few to fill the GPU: the q/k conv and normalisation, which every
    // CTA of a k-head repeats, are then shared by twice the rows (two row
    // slices per head measured 112.6 against 105.4 us per 4-token window at
    // B=128, the work down from 12k to 8.4k warp instructions per 64 rows).
    // For 7 or 8 tokens the rows' longer chain favours more, smaller CTAs
    // (188 against 169 us at 7 tokens with whole heads).
    const int G = s.Hv / s.Hk;
    int SN = (s.T > 6 && s.Dv >= 64 && G * 2 <= 8) ? 2 : 1;
    const long heads = (long)s.B * s.Hv;
    while (SN * 2 <= s.Dv / 16 && G * SN * 2 <= 8 && heads * SN < 2L * num_sms()) SN *= 2;
    WindowParams p{qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, keep, y, err,
                   s.B, s.T, s.Hk, s.Hv, s.Dv, s.C(), s.K, SN, s.eps};
    switch (s.Dk * 8 + s.K) {
        case 32 * 8 + 2: return launch_tm<32, 2>(p, st);
        case 32 * 8 + 3: return launch_tm<32, 3>(p, st);
        case 32 * 8 + 4: return launch_tm<32, 4>(p, st);
        case 64 * 8 + 2: return launch_tm<64, 2>(p, st);
        case 64 * 8 + 3: return launch_tm<64, 3>(p, st);
        case 64 * 8 + 4: return launch_tm<64, 4>(p, st);
        case 128 * 8 + 2: return launch_tm<128, 2>(p, st);
        case 128 * 8 + 3: return launch_tm<128, 3>(p, st);
        case 128 * 8 + 4: return launch_tm<128, 4>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
