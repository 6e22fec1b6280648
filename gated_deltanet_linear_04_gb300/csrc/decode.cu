// One fused decode step: conv window + conv + SiLU + q/k rms-norm, the gates,
// and one step of the gated delta rule, streaming the f32 state once.
//
// Definitions: "mlx-bun 0.4.0 -> 1.0.0, package/src/model/qwen3-delta.ts",
// gated_delta_step (one state row per dv, decay, kv_mem, delta, update, output)
// and computeG; "mlex 0.1.2, src/models/gated_delta.rs", GatedDeltaNet::forward
// (conv window, conv1d + silu, q/k normalisation, beta, g).
//
// HBM-bound design.  A CTA owns R = Dv/SN consecutive rows of one (b, hv)
// state ([Dv, Dk] f32, rows contiguous over Dk).  At entry one thread starts
// 1-D bulk copies (TMA engine) of the whole R x Dk slice into shared memory,
// in 32-row chunks with one mbarrier each, so all of the slice is in flight
// while the CTA computes its conv/norm/gates.  Each chunk is then updated in
// shared memory and the slice written back with one bulk store.
//
// Per row (a group of 8 lanes, each holding Dk/32 of the row's columns as
// float4s; a warp takes four rows at once):
//   sk = S.k                     (3-level shuffle sum)
//   delta = beta (v - g sk)      (kv_mem read from the decayed state g S)
//   S_new = g S + delta k
//   y = S_new . q                (3-level shuffle sum)
// Eight lanes per row instead of a whole warp per row cut the shuffles per
// row from ten to three and need no k.q product (0.869 -> 0.894 of the HBM
// copy peak on the batched-decode workload).
//
// The G = Hv/Hk v-heads of one k-head share the q/k conv channels.  All CTAs of
// one (b, hk) form a thread-block cluster; each reads the old conv_state of
// the q/k channels, arrives on the cluster barrier, and only cluster rank 0
// writes the new q/k conv_state after waiting on it.  v channels belong to one
// CTA each and are updated by it.
//
// NORM variant: the step's output is the layer's RMSNormGated of y ("mlex
// 0.1.2, src/models/gated_delta.rs", GatedDeltaNet::forward: f32 rms_norm of
// the bf16 y over Dv, times the norm weight, times silu(z), cast to bf16)
// instead of y.  It runs only where one CTA holds all Dv rows of a head
// (SN = 1).  With the rows spread over several CTAs the per-head sum needs an
// exchange between them, and every microsecond that adds to a CTA's life
// costs about nine at this occupancy (the state streams through a fixed
// number of CTA slots): measured 115 us per step on the batched-decode
// workload against 102 us for this kernel followed by the separate norm
// kernel, so that pair is used there instead.
#include "common.cuh"
#include "internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kChunkRows = 32;
constexpr int kMaxRows = 128;
constexpr int kMinCtasPerSm = 5;   // launch bound: 48 registers, 5 CTAs of 32 KiB per SM

struct DecodeParams {
    const uint16_t *qkv, *conv_w;
    uint16_t *conv_state;
    const uint16_t *a, *b;
    const float *A_log, *dt_bias;
    float *state;
    const uint8_t *row_mask;
    uint16_t *y;              // y, or the gated-norm output for the NORM variant
    const uint16_t *z;        // NORM: gate input [B, Hv, Dv]
    const float *norm_w;      // NORM: weight [Dv]
    float norm_eps;
    unsigned *err;
    int B, Hk, Hv, Dv, C, K, SN;
    float eps;
};

// Raw inputs of one conv channel: the K-1 stored rows, the new token, the taps.
struct ConvIn {
    uint16_t prev[3];
    uint16_t xnew;
    uint16_t w[4];
};

// the taps (constant across steps) and the step's data, read separately so
// that the taps can be fetched before the wait on the previous step's grid
__device__ __forceinline__ void load_conv_w(const DecodeParams &p, int c, ConvIn &in) {
    const uint16_t *w = p.conv_w + (size_t)c * p.K;
#pragma unroll
    for (int j = 0; j < 4; ++j) in.w[j] = j < p.K ? w[j] : (uint16_t)0;
}

__device__ __forceinline__ void load_conv_data(const DecodeParams &p, int b, int c, ConvIn &in) {
    const int n = p.K - 1;
    const uint16_t *cs = p.conv_state + (size_t)b * n * p.C + c;
#pragma unroll
    for (int j = 0; j < 3; ++j) in.prev[j] = j < n ? cs[(size_t)j * p.C] : (uint16_t)0;
    in.xnew = p.qkv[(size_t)b * p.C + c];
}


// conv over [stored rows, new] followed by SiLU; nw gets the shifted window
// (the new conv_state rows).
__device__ __forceinline__ float conv_apply(int K, const ConvIn &in, uint16_t (&nw)[3]) {
    const int n = K - 1;
    float u = 0.0f;
#pragma unroll
    for (int j = 0; j < 3; ++j)
        if (j < n) u = fmaf(bf16_to_f32(in.w[j]), bf16_to_f32(in.prev[j]), u);
    float wl = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (j == n) wl = bf16_to_f32(in.w[j]);
    u = fmaf(wl, bf16_to_f32(in.xnew), u);
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        if (j < n - 1) nw[j] = in.prev[j + 1];
        else if (j == n - 1) nw[j] = in.xnew;
        else nw[j] = 0;
    }
    return silu(u);
}

template <int DK, bool NORM>
__global__ void __launch_bounds__(kThreads, kMinCtasPerSm) decode_kernel(const DecodeParams p) {
    constexpr int LPR = 8;             // lanes per state row
    constexpr int RPP = 32 / LPR;      // rows per warp pass
    constexpr int NG = DK / 4 / LPR;   // 16-byte column groups per lane
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.Hv / p.Hk;
    const int R = p.Dv / p.SN;
    const int rank = blockIdx.x;      // == %cluster_ctarank (cluster spans grid x)
    const int hv_local = rank / p.SN, slice = rank % p.SN;
    const int hk = blockIdx.y, b = blockIdx.z;
    const int hv = hk * G + hv_local;
    const int r0 = slice * R;
    uint16_t *yrow = p.y + ((size_t)b * p.Hv + hv) * p.Dv + r0;
    grid_dep_launch();

    // before the wait: only the constant taps (and shared-memory set-up below)
    const bool has_qk = tid < 2 * DK;
    const int c_qk = tid < DK ? hk * DK + tid : p.Hk * DK + hk * DK + (tid - DK);
    const bool has_v = tid < R;
    const int c_v = 2 * p.Hk * DK + hv * p.Dv + r0 + tid;
    ConvIn in_qk{}, in_v{};
    if (has_qk) load_conv_w(p, c_qk, in_qk);
    if (has_v) load_conv_w(p, c_v, in_v);
    grid_dep_wait();

    if (p.row_mask != nullptr && p.row_mask[b] == 0) {
        // whole cluster shares b: every CTA leaves here, no barrier is pending
        for (int i = tid; i < R; i += kThreads) yrow[i] = 0;
        return;
    }

    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *S = reinterpret_cast<float *>(smem_raw);
    __shared__ __align__(16) float q_s[DK];
    __shared__ __align__(16) float k_s[DK];
    __shared__ float v_s[kMaxRows];
    __shared__ float y_s[kMaxRows];
    __shared__ float red[kThreads / 32];
    __shared__ float gbk[2];                       // g, beta
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

    // ---- conv + SiLU for the q/k channels of hk and the v channels of the slice
    uint16_t nw_qk[3] = {0, 0, 0}, nw_v[3] = {0, 0, 0};
    float xqk = 0.0f;
    // all raw conv inputs of both channels in flight before any arithmetic
    if (has_qk) load_conv_data(p, b, c_qk, in_qk);
    if (has_v) load_conv_data(p, b, c_v, in_v);
    if (has_qk) xqk = conv_apply(p.K, in_qk, nw_qk);
    if (has_v) v_s[tid] = round_bf16(conv_apply(p.K, in_v, nw_v));
    // NORM: z and the weight of this thread's row, fetched now so that their
    // latency hides behind the state copy
    float zv = 0.0f, wv = 0.0f;
    if constexpr (NORM) {
        if (tid < R) {
            zv = bf16_to_f32(p.z[((size_t)b * p.Hv + hv) * p.Dv + r0 + tid]);
            wv = p.norm_w[r0 + tid];
        }
    }
    // every read of the shared (q/k) conv_state of this CTA has been consumed
    // above, so a relaxed arrive suffices (a release arrive would also wait for
    // this thread's unrelated outstanding accesses)
    cluster_arrive_relaxed();

    // rms-norm sums: q channels are threads [0, DK), k channels [DK, 2 DK)
    float ss = warp_sum(has_qk ? xqk * xqk : 0.0f);
    if (lane == 0) red[warp] = ss;
    if (tid == 0) {
        const float x = bf16_to_f32(p.a[(size_t)b * p.Hv + hv]) + p.dt_bias[hv];
        gbk[0] = expf(-expf(p.A_log[hv]) * softplus(x));
        gbk[1] = sigmoid(bf16_to_f32(p.b[(size_t)b * p.Hv + hv]));
    }
    __syncthreads();
    if (has_qk) {
        constexpr int NW = DK / 32;
        const bool is_q = tid < DK;
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) tot += red[(is_q ? 0 : NW) + w];
        const float inv_d = 1.0f / (float)DK;
        const float scale = is_q ? inv_d : 1.0f / sqrtf((float)DK);
        const float val = round_bf16(xqk * ((1.0f / sqrtf(tot * inv_d + p.eps)) * scale));
        if (is_q) q_s[tid] = val;
        else k_s[tid - DK] = val;
    }
    __syncthreads();

    // ---- the recurrence step over the state slice: eight lanes per row
    // (lane l holds the row's 16-byte column groups l, l + 8, ..., so a
    // quarter-warp's shared-memory accesses fall on distinct banks); S' k,
    // the update, then y = S q
    const int sub = lane / LPR, cl = lane % LPR;
    const float4 *k4 = reinterpret_cast<const float4 *>(k_s);
    const float4 *q4 = reinterpret_cast<const float4 *>(q_s);
    const float g = gbk[0], beta = gbk[1];
    bool ok_all = true;
    for (int p0 = warp * RPP; p0 < R; p0 += (kThreads / 32) * RPP) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[p0 / rc], 0, p.err));
        ok_all = ok_all && ok;
        if (!ok) continue;
        const int ra = p0 + sub;
        float4 *spa = reinterpret_cast<float4 *>(S + (size_t)ra * DK);
        float4 sa[NG];
#pragma unroll
        for (int j = 0; j < NG; ++j) sa[j] = spa[j * LPR + cl];
        // column pairs on the packed two-wide f32 instructions (each half
        // rounds like the scalar one; the pair's halves are the two partial
        // sums of the row's dot products)
        float2 pa = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const float4 kk = k4[j * LPR + cl];
            pa = __ffma2_rn(make_float2(sa[j].x, sa[j].y), make_float2(kk.x, kk.y), pa);
            pa = __ffma2_rn(make_float2(sa[j].z, sa[j].w), make_float2(kk.z, kk.w), pa);
        }
        float dka = pa.x + pa.y;
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) dka += __shfl_xor_sync(0xffffffffu, dka, o);
        const float da = beta * (v_s[ra] - g * dka);
        const float2 g2 = make_float2(g, g), da2 = make_float2(da, da);
        pa = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const float4 kk = k4[j * LPR + cl];
            const float2 lo = __ffma2_rn(da2, make_float2(kk.x, kk.y), __fmul2_rn(g2, make_float2(sa[j].x, sa[j].y)));
            const float2 hi = __ffma2_rn(da2, make_float2(kk.z, kk.w), __fmul2_rn(g2, make_float2(sa[j].z, sa[j].w)));
            sa[j] = make_float4(lo.x, lo.y, hi.x, hi.y);
            spa[j * LPR + cl] = sa[j];
            const float4 qq = q4[j * LPR + cl];
            pa = __ffma2_rn(lo, make_float2(qq.x, qq.y), pa);
            pa = __ffma2_rn(hi, make_float2(qq.z, qq.w), pa);
        }
        float dqa = pa.x + pa.y;
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) dqa += __shfl_xor_sync(0xffffffffu, dqa, o);
        if (cl == 0) y_s[ra] = dqa;
    }
    fence_proxy_async_smem();
    ok_all = __syncthreads_and(ok_all) != 0;
    if (ok_all && tid == 0) {
        bulk_store(gstate, S, (uint32_t)R * DK * 4);
        bulk_commit();
    }

    if constexpr (!NORM) {
        if (ok_all)
            for (int i = tid; i < R; i += kThreads) yrow[i] = f32_to_bf16(y_s[i]);
    } else {
        // gated RMS norm of the head's bf16 y over all Dv rows
        const float yv = tid < R ? round_bf16(y_s[tid]) : 0.0f;
        const float ss = warp_sum(yv * yv);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) tot += red[w];
        if (tid < R && ok_all) {
            const float rs = 1.0f / sqrtf(tot * (1.0f / (float)p.Dv) + p.norm_eps);
            yrow[tid] = f32_to_bf16(silu(zv) * ((yv * rs) * wv));
        }
    }

    // ---- new conv_state: rank 0 writes the shared q/k channels after every
    // CTA of the cluster has read them; each CTA writes its own v channels.
    cluster_wait_acquire();
    const int n = p.K - 1;
    if (has_qk && rank == 0) {
        uint16_t *cs = p.conv_state + (size_t)b * n * p.C + c_qk;
        for (int j = 0; j < n; ++j) cs[(size_t)j * p.C] = nw_qk[j];
    }
    if (has_v) {
        uint16_t *cs = p.conv_state + (size_t)b * n * p.C + c_v;
        for (int j = 0; j < n; ++j) cs[(size_t)j * p.C] = nw_v[j];
    }
    if (tid == 0) bulk_wait_read();   // the slice has been read out of shared memory
}

template <int DK, bool NORM>
cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t st) {
    const int G = p.Hv / p.Hk;
    const int R = p.Dv / p.SN;
    const size_t smem = (size_t)R * DK * sizeof(float);
    static unsigned long long attr_done = 0;   // per instantiation, one bit per device
    cudaError_t ae = once_per_device(attr_done, [] {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<DK, NORM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(kMaxRows * DK * sizeof(float)));
        if (e != cudaSuccess) return e;
        return cudaFuncSetAttribute(decode_kernel<DK, NORM>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    });
    if (ae != cudaSuccess) return ae;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G * p.SN, p.Hk, p.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G * p.SN;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // Programmatic launch pays when the grid spans several waves (the next
    // step's CTAs fill SMs as this grid's tail drains: 0.855 -> 0.868 of the
    // HBM copy peak at B=128); a grid that fits in one resident wave gains
    // nothing and its wait is slower than a plain graph edge (4.69 -> 5.73
    // us per B=1 step in a CUDA graph), so it launches without it.
    const long ctas = (long)cfg.gridDim.x * cfg.gridDim.y * cfg.gridDim.z;
    cfg.numAttrs = ctas > (long)kMinCtasPerSm * num_sms() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel<DK, NORM>, p);
}

}  // namespace

cudaError_t launch_decode(const Sizes &s, const uint16_t *qkv, const uint16_t *conv_w, uint16_t *conv_state,
                          const uint16_t *a, const uint16_t *b, const float *A_log, const float *dt_bias,
                          float *state, const uint8_t *row_mask, uint16_t *y, const uint16_t *z,
                          const float *norm_w, float norm_eps, unsigned *err, cudaStream_t st) {
    const int G = s.Hv / s.Hk;
    // Split each head's rows over SN CTAs: at least 2 when rows allow (smaller
    // CTAs keep more of them, at different phases, resident per SM: measured
    // 0.83 vs 0.74 of the HBM copy peak on the batched-decode workload), more
    // until the grid covers the GPU twice; >= 16 rows per CTA and clusters of
    // at most 8 CTAs (16 if G = 16).
    int SN = (s.Dv >= 64 && G * 2 <= 8) ? 2 : 1;
    const long heads = (long)s.B * s.Hv;
    while (SN * 2 <= s.Dv / 16 && G * SN * 2 <= 8 && heads * SN < 2L * num_sms()) SN *= 2;
    DecodeParams p{qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, row_mask, y, z, norm_w, norm_eps, err,
                   s.B, s.Hk, s.Hv, s.Dv, s.C(), s.K, SN, s.eps};
    const bool norm = z != nullptr && SN == 1;
    if (z != nullptr && SN > 1) {
        // rows of a head over several CTAs: y into the output, then the norm in place
        cudaError_t e = cudaSuccess;
        switch (s.Dk) {
            case 32: e = launch_decode_t<32, false>(p, st); break;
            case 64: e = launch_decode_t<64, false>(p, st); break;
            case 128: e = launch_decode_t<128, false>(p, st); break;
            default: return cudaErrorInvalidValue;
        }
        if (e != cudaSuccess) return e;
        return launch_rmsnorm_gated(s, y, z, norm_w, norm_eps, y, st);
    }
    switch (s.Dk) {
        case 32: return norm ? launch_decode_t<32, true>(p, st) : launch_decode_t<32, false>(p, st);
        case 64: return norm ? launch_decode_t<64, true>(p, st) : launch_decode_t<64, false>(p, st);
        case 128: return norm ? launch_decode_t<128, true>(p, st) : launch_decode_t<128, false>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
