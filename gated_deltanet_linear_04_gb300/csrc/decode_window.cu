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
// Same layout as the single-token kernel: a cluster per (b, hk) group of the
// G v-heads x SN row slices, each CTA bulk-copies its R x Dk state slice into
// shared memory while it computes the conv/norm/gates of the T tokens.  Eight
// lanes walk a row through all T tokens with the row in registers (a warp
// takes four rows at once, so a row's dot products are 3-level shuffle sums;
// lane l holds the row's 16-byte column groups l, l + 8, ..., which keeps
// each quarter-warp's shared-memory accesses on distinct banks); after token
// keep-1 the row is written back to shared memory, so the slice stored at the
// end is the state after the kept prefix (nothing is stored when keep is 0).
#include "common.cuh"
#include "internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
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

// SiLU(conv) of the T new tokens of channel c.  The window is held as
// x[0 .. K-1) = the stored rows (oldest first) and x[K-1 + t] = token t, so
// token t's taps j = 0 .. K-1 read x[t + j] (its own value on tap K-1).
template <int K>
__device__ __forceinline__ void conv_tokens(const WindowParams &p, int b, int c, float (&out)[kMaxT]) {
    constexpr int n = K - 1;
    float x[n + kMaxT];
    const uint16_t *cs = p.conv_state + (size_t)b * n * p.C + c;
#pragma unroll
    for (int j = 0; j < n; ++j) x[j] = bf16_to_f32(cs[(size_t)j * p.C]);
#pragma unroll
    for (int t = 0; t < kMaxT; ++t)
        x[n + t] = t < p.T ? bf16_to_f32(p.qkv[((size_t)b * p.T + t) * p.C + c]) : 0.0f;
    float w[K];
#pragma unroll
    for (int j = 0; j < K; ++j) w[j] = bf16_to_f32(p.conv_w[(size_t)c * K + j]);
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
        float u = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) u = fmaf(w[j], x[t + j], u);
        out[t] = silu(u);
    }
}

// conv_state of channel c after the first `keep` (>= 1) tokens: row j is
// window entry keep + j, i.e. stored row keep + j while that is < K-1, else
// token keep + j - (K-1).  Rows are written in increasing j, and row j reads
// a stored row > j, so the rows it reads are still the old ones.
template <int K>
__device__ __forceinline__ void write_conv_state(const WindowParams &p, int b, int c, int keep) {
    constexpr int n = K - 1;
    uint16_t *cs = p.conv_state + (size_t)b * n * p.C + c;
#pragma unroll
    for (int j = 0; j < n; ++j) {
        const int pos = keep + j;
        const uint16_t v = pos < n ? cs[(size_t)pos * p.C] : p.qkv[((size_t)b * p.T + (pos - n)) * p.C + c];
        cs[(size_t)j * p.C] = v;
    }
}

template <int DK, int K>
__global__ void __launch_bounds__(kThreads, 4) window_kernel(const WindowParams p) {
    constexpr int LPR = 8;             // lanes per row
    constexpr int RPP = 32 / LPR;      // rows per warp pass
    constexpr int NG = DK / 4 / LPR;   // 16-byte column groups per lane
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.Hv / p.Hk;
    const int R = p.Dv / p.SN;
    const int rank = blockIdx.x;
    const int hv_local = rank / p.SN, slice = rank % p.SN;
    const int hk = blockIdx.y, b = blockIdx.z;
    const int hv = hk * G + hv_local;
    const int r0 = slice * R;
    const int T = p.T;
    int keep = p.keep == nullptr ? T : p.keep[b];
    keep = keep < 0 ? 0 : (keep > T ? T : keep);

    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *S = reinterpret_cast<float *>(smem_raw);
    __shared__ __align__(16) float q_s[kMaxT][DK];
    __shared__ __align__(16) float k_s[kMaxT][DK];
    __shared__ float v_s[kMaxT][kMaxRows];
    __shared__ float y_s[kMaxT][kMaxRows];
    __shared__ float red[kMaxT][kThreads / 32];
    __shared__ float gq[kMaxT][3];                 // g, beta, k.q per token
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

    // ---- conv + SiLU of the T tokens: q/k channels of hk, v channels of the slice
    const bool has_qk = tid < 2 * DK;
    const int c_qk = tid < DK ? hk * DK + tid : p.Hk * DK + hk * DK + (tid - DK);
    const bool has_v = tid < R;
    const int c_v = 2 * p.Hk * DK + hv * p.Dv + r0 + tid;
    float xqk[kMaxT];
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) xqk[t] = 0.0f;
    if (has_qk) conv_tokens<K>(p, b, c_qk, xqk);
    if (has_v) {
        float xv[kMaxT];
        conv_tokens<K>(p, b, c_v, xv);
#pragma unroll
        for (int t = 0; t < kMaxT; ++t)
            if (t < T) v_s[t][tid] = round_bf16(xv[t]);
    }
#pragma unroll
    for (int t = 0; t < kMaxT; ++t)
        if (t >= T) xqk[t] = 0.0f;
    cluster_arrive_relaxed();      // the shared q/k conv_state has been read
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
        if (t < T) {
            const float ss = warp_sum(xqk[t] * xqk[t]);
            if (lane == 0) red[t][warp] = ss;
        }
    }
    if (tid < T) {
        const size_t gi = ((size_t)b * T + tid) * p.Hv + hv;
        const float x = bf16_to_f32(p.a[gi]) + p.dt_bias[hv];
        gq[tid][0] = expf(-expf(p.A_log[hv]) * softplus(x));
        gq[tid][1] = sigmoid(bf16_to_f32(p.b[gi]));
    }
    __syncthreads();
    if (has_qk) {
        constexpr int NW = DK / 32;
        const bool is_q = tid < DK;
        const float inv_d = 1.0f / (float)DK;
        const float scale = is_q ? inv_d : 1.0f / sqrtf((float)DK);
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) {
            if (t < T) {
                float tot = 0.0f;
#pragma unroll
                for (int w = 0; w < NW; ++w) tot += red[t][(is_q ? 0 : NW) + w];
                const float val = round_bf16(xqk[t] * ((1.0f / sqrtf(tot * inv_d + p.eps)) * scale));
                if (is_q) q_s[t][tid] = val;
                else k_s[t][tid - DK] = val;
            }
        }
    }
    __syncthreads();
    if (warp < T) {
        float kq = 0.0f;
        for (int i = lane; i < DK; i += 32) kq = fmaf(k_s[warp][i], q_s[warp][i], kq);
        kq = warp_sum(kq);
        if (lane == 0) gq[warp][2] = kq;
    }
    __syncthreads();

    // ---- rows through the window
    const int sub = lane / LPR, cl = lane % LPR;
    bool ok_all = true;
    for (int ch = 0; ch < nch; ++ch) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[ch], 0, p.err));
        ok_all = ok_all && ok;
        if (!ok) continue;
        for (int rr = warp * RPP + sub; rr < rc; rr += (kThreads / 32) * RPP) {
            const int row = ch * rc + rr;
            float4 *sp = reinterpret_cast<float4 *>(S + (size_t)row * DK);
            float4 s[NG];
#pragma unroll
            for (int j = 0; j < NG; ++j) s[j] = sp[j * LPR + cl];
            for (int t = 0; t < T; ++t) {
                const float4 *k4 = reinterpret_cast<const float4 *>(k_s[t]);
                const float4 *q4 = reinterpret_cast<const float4 *>(q_s[t]);
                const float g = gq[t][0], beta = gq[t][1], kq = gq[t][2];
                float dk0 = 0.0f, dk1 = 0.0f, dq0 = 0.0f, dq1 = 0.0f;
#pragma unroll
                for (int j = 0; j < NG; ++j) {
                    const float4 kk = k4[j * LPR + cl], qq = q4[j * LPR + cl];
                    dk0 = fmaf(s[j].x, kk.x, dk0);
                    dk1 = fmaf(s[j].y, kk.y, dk1);
                    dk0 = fmaf(s[j].z, kk.z, dk0);
                    dk1 = fmaf(s[j].w, kk.w, dk1);
                    dq0 = fmaf(s[j].x, qq.x, dq0);
                    dq1 = fmaf(s[j].y, qq.y, dq1);
                    dq0 = fmaf(s[j].z, qq.z, dq0);
                    dq1 = fmaf(s[j].w, qq.w, dq1);
                }
                float dk = dk0 + dk1, dq = dq0 + dq1;
#pragma unroll
                for (int o = LPR / 2; o > 0; o >>= 1) {
                    dk += __shfl_xor_sync(0xffffffffu, dk, o);
                    dq += __shfl_xor_sync(0xffffffffu, dq, o);
                }
                const float delta = beta * (v_s[t][row] - g * dk);
#pragma unroll
                for (int j = 0; j < NG; ++j) {
                    const float4 kk = k4[j * LPR + cl];
                    s[j].x = fmaf(delta, kk.x, g * s[j].x);
                    s[j].y = fmaf(delta, kk.y, g * s[j].y);
                    s[j].z = fmaf(delta, kk.z, g * s[j].z);
                    s[j].w = fmaf(delta, kk.w, g * s[j].w);
                }
                if (cl == 0) y_s[t][row] = fmaf(delta, kq, g * dq);
                if (t == keep - 1) {              // the state after the kept prefix
#pragma unroll
                    for (int j = 0; j < NG; ++j) sp[j * LPR + cl] = s[j];
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
    if (ok_all)
        for (int i = tid; i < T * R; i += kThreads) {
            const int t = i / R, r = i % R;
            p.y[(((size_t)b * T + t) * p.Hv + hv) * p.Dv + r0 + r] = f32_to_bf16(y_s[t][r]);
        }

    // ---- conv_state after the kept prefix: rank 0 writes the shared q/k
    // channels once every CTA of the cluster has read them
    cluster_wait_acquire();
    if (keep > 0) {
        if (has_qk && rank == 0) write_conv_state<K>(p, b, c_qk, keep);
        if (has_v) write_conv_state<K>(p, b, c_v, keep);
    }
    if (tid == 0) bulk_wait_read();   // the slice has been read out of shared memory
}

template <int DK, int K>
cudaError_t launch_t(const WindowParams &p, cudaStream_t st) {
    const int G = p.Hv / p.Hk;
    const int R = p.Dv / p.SN;
    static unsigned long long attr_done = 0;   // per instantiation, one bit per device
    cudaError_t ae = once_per_device(attr_done, [] {
        cudaError_t e = cudaFuncSetAttribute(window_kernel<DK, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(kMaxRows * DK * sizeof(float)));
        if (e != cudaSuccess) return e;
        return cudaFuncSetAttribute(window_kernel<DK, K>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    });
    if (ae != cudaSuccess) return ae;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G * p.SN, p.Hk, p.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)R * DK * sizeof(float);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G * p.SN;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, window_kernel<DK, K>, p);
}

}  // namespace

cudaError_t launch_decode_window(const Sizes &s, const uint16_t *qkv, const uint16_t *conv_w, uint16_t *conv_state,
                                 const uint16_t *a, const uint16_t *b, const float *A_log, const float *dt_bias,
                                 float *state, const int32_t *keep, uint16_t *y, unsigned *err, cudaStream_t st) {
    if (s.T < 1 || s.T > kMaxT) return cudaErrorNotSupported;
    const int G = s.Hv / s.Hk;
    int SN = (s.Dv >= 64 && G * 2 <= 8) ? 2 : 1;
    const long heads = (long)s.B * s.Hv;
    while (SN * 2 <= s.Dv / 16 && G * SN * 2 <= 8 && heads * SN < 2L * num_sms()) SN *= 2;
    WindowParams p{qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, keep, y, err,
                   s.B, s.T, s.Hk, s.Hv, s.Dv, s.C(), s.K, SN, s.eps};
    switch (s.Dk * 8 + s.K) {
        case 32 * 8 + 2: return launch_t<32, 2>(p, st);
        case 32 * 8 + 3: return launch_t<32, 3>(p, st);
        case 32 * 8 + 4: return launch_t<32, 4>(p, st);
        case 64 * 8 + 2: return launch_t<64, 2>(p, st);
        case 64 * 8 + 3: return launch_t<64, 3>(p, st);
        case 64 * 8 + 4: return launch_t<64, 4>(p, st);
        case 128 * 8 + 2: return launch_t<128, 2>(p, st);
        case 128 * 8 + 3: return launch_t<128, 3>(p, st);
        case 128 * 8 + 4: return launch_t<128, 4>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
