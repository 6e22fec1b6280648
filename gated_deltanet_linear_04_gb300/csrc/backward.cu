// Backward pass of the recurrence (sequential form): the gradients of y and of
// the final state with respect to q, k, v, g, beta and the initial state.
//
// The pages ("mlex 0.1.2, src/models/gated_delta.rs", the per-timestep loop;
// "mlx-bun 0.4.0 -> 1.0.0, package/src/model/qwen3-delta.ts",
// gated_delta_step) define the forward step only; this is its exact
// derivative, taken step by step in reverse.  With S' = g_t S_{t-1},
// u = v_t - S' k_t, delta = beta_t u, S_t = S' + delta k_t^T, y_t = S_t q_t
// and dS the gradient of S_t:
//   dS += dy_t q_t^T            dq_t = S_t^T dy_t
//   ddelta = dS k_t             dk_t = dS^T delta
//   dbeta_t = ddelta . u        du = beta_t ddelta        dv_t = du
//   dS' = dS - du k_t^T         dk_t -= S'^T du
//   dg_t = <dS', S_{t-1}>       dS_{t-1} = g_t dS'
// A masked step has zero gradients for its inputs and passes dS through.
//
// Work split: a CTA (4 warps) owns 32 state rows of one (b, hv) head; lane
// (rg, cg) of warp w holds rows w*8 + rg*2 + {0, 1} and columns
// [cg*Dk/8, (cg+1)*Dk/8), so a row's dot product is a 3-level shuffle sum over
// the 8 lanes sharing rg.  The rows of the state evolve independently, so
// the slice first runs the forward recurrence storing its rows every 32 steps
// (checkpoints), then walks the chunks of 32 steps backwards: it recomputes
// the chunk's states from the checkpoint into a history buffer (global memory,
// L2-resident) keeping u per row, and runs the reverse steps with dS in
// registers.  The sums over rows (dq, dk, dg, dbeta) are reduced within the
// warp, collected per step in shared memory and added to the outputs with
// atomics once per chunk; the atomics also sum over the row slices and over
// the v-heads that share a k-head.  The call zeroes the outputs first.
#include "common.cuh"
#include "internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 128;
constexpr int kRows = 32;        // state rows per CTA
constexpr int kC = 32;           // steps per chunk / checkpoint interval

struct BwdParams {
    const uint16_t *q, *k, *v;
    const float *g, *beta, *state_in;
    const uint8_t *mask;
    const uint16_t *dy;
    const float *dstate_out;
    float *dq, *dk, *dv, *dg, *dbeta, *dstate_in;
    float *ws;
    int B, T, Hk, Hv, Dv, nck;
};

template <int DK>
struct BwdSmem {
    float q[kC][DK], k[kC][DK];
    float v[kC][kRows], dy[kC][kRows], u[kC][kRows];
    float g[kC], beta[kC];
    int m[kC];
    float red_q[kC][DK], red_k[kC][DK];
    float red_g[kC], red_b[kC];
};

// Stage steps [t0, t0 + n) of the chunk: q, k of the k-head, v and dy of the
// CTA's rows, g, beta, the mask (steps past T or masked: m = 0).  Block-wide;
// ends with a barrier.  with_q_dy = false for the forward sweep.
template <int DK>
__device__ __forceinline__ void stage_chunk(const BwdParams &p, BwdSmem<DK> &s, int b, int hk, int hv, int r0,
                                            int t0, bool with_q_dy) {
    const int tid = threadIdx.x;
    const int T = p.T;
    constexpr int V8 = DK / 8;   // 16-byte groups of a q / k row
    for (int i = tid; i < kC * V8; i += kThreads) {
        const int tl = i / V8, c8 = (i % V8) * 8, t = t0 + tl;
        uint4 kk = make_uint4(0u, 0u, 0u, 0u), qq = kk;
        if (t < T) {
            const size_t off = (((size_t)b * T + t) * p.Hk + hk) * DK + c8;
            kk = *reinterpret_cast<const uint4 *>(p.k + off);
            if (with_q_dy) qq = *reinterpret_cast<const uint4 *>(p.q + off);
        }
        const uint32_t kw[4] = {kk.x, kk.y, kk.z, kk.w}, qw[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s.k[tl][c8 + 2 * e] = __uint_as_float(kw[e] << 16);
            s.k[tl][c8 + 2 * e + 1] = __uint_as_float(kw[e] & 0xffff0000u);
            s.q[tl][c8 + 2 * e] = __uint_as_float(qw[e] << 16);
            s.q[tl][c8 + 2 * e + 1] = __uint_as_float(qw[e] & 0xffff0000u);
        }
    }
    for (int i = tid; i < kC * kRows; i += kThreads) {
        const int tl = i / kRows, r = i % kRows, t = t0 + tl;
        float vv = 0.0f, dd = 0.0f;
        if (t < T) {
            const size_t off = (((size_t)b * T + t) * p.Hv + hv) * p.Dv + r0 + r;
            vv = bf16_to_f32(p.v[off]);
            if (with_q_dy) dd = bf16_to_f32(p.dy[off]);
        }
        s.v[tl][r] = vv;
        s.dy[tl][r] = dd;
    }
    if (tid < kC) {
        const int t = t0 + tid;
        int m = 0;
        float gg = 1.0f, bb = 0.0f;
        if (t < T) {
            m = p.mask == nullptr ? 1 : (p.mask[(size_t)b * T + t] != 0);
            const size_t gi = ((size_t)b * T + t) * p.Hv + hv;
            gg = p.g[gi];
            bb = p.beta[gi];
        }
        s.m[tid] = m;
        s.g[tid] = gg;
        s.beta[tid] = bb;
    }
    __syncthreads();
}

// Whether steps [t0, t0 + kC) of row b hold a valid step (uniform over the CTA).
__device__ __forceinline__ bool chunk_active(const BwdParams &p, int b, int t0) {
    if (p.mask == nullptr) return true;
    const int t = t0 + (int)threadIdx.x;
    const bool m = threadIdx.x < kC && t < p.T && p.mask[(size_t)b * p.T + t] != 0;
    return __syncthreads_or(m) != 0;
}

// sum over the 8 lanes of a row group (lanes differing in bits 0-2)
__device__ __forceinline__ float row_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
}

template <int DK>
__global__ void __launch_bounds__(kThreads) backward_kernel(const BwdParams p) {
    constexpr int CW = DK / 8;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<DK> &s = *reinterpret_cast<BwdSmem<DK> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = lane >> 3, cg = lane & 7;
    const int slice = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
    const int hk = hv / (p.Hv / p.Hk);
    const int r0 = slice * kRows;
    const int T = p.T;
    const int c0 = cg * CW;
    int rl[2];
    rl[0] = warp * 8 + rg * 2;
    rl[1] = rl[0] + 1;
    const size_t head = (size_t)b * p.Hv + hv;
    // this CTA's checkpoints [nck][kRows][DK] and chunk history [kC][kRows][DK]
    const size_t cta = head * (p.Dv / kRows) + slice;
    float *ck = p.ws + cta * (size_t)(p.nck + kC) * kRows * DK;
    float *hist = ck + (size_t)p.nck * kRows * DK;

    auto load_rows = [&](const float *src, float (&x)[2][CW]) {   // src: [kRows][DK]
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < CW; j += 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(src + (size_t)rl[i] * DK + c0 + j);
                x[i][j] = v4.x; x[i][j + 1] = v4.y; x[i][j + 2] = v4.z; x[i][j + 3] = v4.w;
            }
    };
    auto store_rows = [&](float *dst, const float (&x)[2][CW]) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < CW; j += 4)
                *reinterpret_cast<float4 *>(dst + (size_t)rl[i] * DK + c0 + j) =
                    make_float4(x[i][j], x[i][j + 1], x[i][j + 2], x[i][j + 3]);
    };
    // one forward step of the two rows from the staged chunk; returns u per row
    auto fwd_step = [&](float (&S)[2][CW], int tl, float (&u)[2]) {
        const float gg = s.g[tl], bb = s.beta[tl];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float kv = 0.0f;
#pragma unroll
            for (int j = 0; j < CW; ++j) kv = fmaf(S[i][j], s.k[tl][c0 + j], kv);
            kv = gg * row_sum(kv);
            u[i] = s.v[tl][rl[i]] - kv;
            const float dl = bb * u[i];
#pragma unroll
            for (int j = 0; j < CW; ++j) S[i][j] = fmaf(dl, s.k[tl][c0 + j], gg * S[i][j]);
        }
    };

    float S[2][CW];
    if (p.state_in != nullptr) {
        load_rows(p.state_in + (head * p.Dv + r0) * DK, S);
    } else {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < CW; ++j) S[i][j] = 0.0f;
    }

    // ---- forward sweep: checkpoint every kC steps
    for (int c = 0; c < p.nck; ++c) {
        store_rows(ck + (size_t)c * kRows * DK, S);
        if (!chunk_active(p, b, c * kC)) continue;   // the identity on the state
        stage_chunk<DK>(p, s, b, hk, hv, r0, c * kC, false);
        for (int tl = 0; tl < kC; ++tl) {
            if (!s.m[tl]) continue;
            float u[2];
            fwd_step(S, tl, u);
        }
        __syncthreads();
    }

    // ---- reverse sweep
    float dS[2][CW];
    if (p.dstate_out != nullptr) {
        load_rows(p.dstate_out + (head * p.Dv + r0) * DK, dS);
    } else {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < CW; ++j) dS[i][j] = 0.0f;
    }
    for (int c = p.nck - 1; c >= 0; --c) {
        const int t0 = c * kC;
        if (!chunk_active(p, b, t0)) continue;   // dS passes through; its gradients stay zero
        stage_chunk<DK>(p, s, b, hk, hv, r0, t0, true);
        for (int i = tid; i < kC * DK; i += kThreads) {
            (&s.red_q[0][0])[i] = 0.0f;
            (&s.red_k[0][0])[i] = 0.0f;
        }
        if (tid < kC) {
            s.red_g[tid] = 0.0f;
            s.red_b[tid] = 0.0f;
        }
        // recompute the chunk: hist[tl] = the state before step tl
        load_rows(ck + (size_t)c * kRows * DK, S);
        for (int tl = 0; tl < kC; ++tl) {
            store_rows(hist + (size_t)tl * kRows * DK, S);
            if (!s.m[tl]) continue;
            float u[2];
            fwd_step(S, tl, u);
            if (cg == 0) {
                s.u[tl][rl[0]] = u[0];
                s.u[tl][rl[1]] = u[1];
            }
        }
        __syncthreads();
        // S is now the state after the chunk; walk it backwards, the state
        // before each step read from the history one step ahead
        float Sp[2][CW];
        load_rows(hist + (size_t)(kC - 1) * kRows * DK, Sp);
        for (int tl = kC - 1; tl >= 0; --tl) {
            float Sn[2][CW];   // S_{t-2}, for the next reverse step
            if (tl > 0) load_rows(hist + (size_t)(tl - 1) * kRows * DK, Sn);
            if (s.m[tl]) {
                const float gg = s.g[tl], bb = s.beta[tl];
                float dq_p[CW], dk_p[CW];
#pragma unroll
                for (int j = 0; j < CW; ++j) dq_p[j] = dk_p[j] = 0.0f;
                float dg_p = 0.0f, db_p = 0.0f;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float dyv = s.dy[tl][rl[i]];
                    const float ui = s.u[tl][rl[i]];
                    float dd = 0.0f;
#pragma unroll
                    for (int j = 0; j < CW; ++j) {
                        dS[i][j] = fmaf(dyv, s.q[tl][c0 + j], dS[i][j]);
                        dq_p[j] = fmaf(S[i][j], dyv, dq_p[j]);
                        dd = fmaf(dS[i][j], s.k[tl][c0 + j], dd);
                    }
                    dd = row_sum(dd);                       // ddelta of the row
                    const float dl = bb * ui;               // delta
                    const float du = bb * dd;
                    if (cg == 0) {
                        db_p = fmaf(dd, ui, db_p);
                        p.dv[(((size_t)b * T + t0 + tl) * p.Hv + hv) * p.Dv + r0 + rl[i]] = du;
                    }
#pragma unroll
                    for (int j = 0; j < CW; ++j) {
                        dk_p[j] = fmaf(dS[i][j], dl, dk_p[j]);
                        dS[i][j] = fmaf(-du, s.k[tl][c0 + j], dS[i][j]);
                        dk_p[j] = fmaf(-gg * Sp[i][j], du, dk_p[j]);
                        dg_p = fmaf(dS[i][j], Sp[i][j], dg_p);
                        dS[i][j] *= gg;
                    }
                }
                // sum the 2*CW partials (dq, dk) over the warp's four row
                // groups in two exchanges that halve the vector: lanes whose
                // rg differs in bit 0 swap halves (dq <-> dk), then lanes whose
                // rg differs in bit 1 swap quarters, so each lane ends with
                // CW/2 summed columns (of dq for even rg, dk for odd) and adds
                // those; the pairwise sums are those of a per-column shuffle sum
                const bool hi0 = (rg & 1) != 0, hi1 = (rg & 2) != 0;
                float h[CW];
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    const float send = hi0 ? dq_p[j] : dk_p[j];
                    const float keep = hi0 ? dk_p[j] : dq_p[j];
                    h[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                constexpr int HQ = CW / 2;
                float *dst = (hi0 ? &s.red_k[tl][c0] : &s.red_q[tl][c0]) + (hi1 ? HQ : 0);
#pragma unroll
                for (int j = 0; j < HQ; ++j) {
                    const float send = hi1 ? h[j] : h[HQ + j];
                    const float keep = hi1 ? h[HQ + j] : h[j];
                    atomicAdd(dst + j, keep + __shfl_xor_sync(0xffffffffu, send, 16));
                }
                dg_p = warp_sum(dg_p);
                db_p = warp_sum(db_p);
                if (lane == 0) {
                    atomicAdd(&s.red_g[tl], dg_p);
                    atomicAdd(&s.red_b[tl], db_p);
                }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    S[i][j] = Sp[i][j];
                    Sp[i][j] = Sn[i][j];
                }
        }
        __syncthreads();
        // add the chunk's sums to the outputs (also summing over row slices
        // and over the v-heads of the k-head)
        const int n = min(kC, T - t0);
        for (int i = tid; i < n * DK; i += kThreads) {
            const int tl = i / DK, j = i % DK;
            if (!s.m[tl]) continue;
            const size_t o = (((size_t)b * T + t0 + tl) * p.Hk + hk) * DK + j;
            atomicAdd(p.dq + o, s.red_q[tl][j]);
            atomicAdd(p.dk + o, s.red_k[tl][j]);
        }
        if (tid < n && s.m[tid]) {
            const size_t o = ((size_t)b * T + t0 + tid) * p.Hv + hv;
            atomicAdd(p.dg + o, s.red_g[tid]);
            atomicAdd(p.dbeta + o, s.red_b[tid]);
        }
        __syncthreads();
    }
    store_rows(p.dstate_in + (head * p.Dv + r0) * DK, dS);
}

template <int DK>
cudaError_t launch_bwd_t(const Sizes &s, const BwdParams &p, cudaStream_t st) {
    const size_t smem = sizeof(BwdSmem<DK>);
    static unsigned long long attr_done = 0;   // per instantiation, one bit per device
    cudaError_t e = set_max_smem(attr_done, backward_kernel<DK>, smem);
    if (e != cudaSuccess) return e;
    backward_kernel<DK><<<dim3(s.Dv / kRows, s.Hv, s.B), kThreads, smem, st>>>(p);
    return cudaGetLastError();
}

size_t nck_of(const Sizes &s) { return ((size_t)s.T + kC - 1) / kC; }

}  // namespace

size_t backward_workspace(const Sizes &s) {
    const size_t ctas = (size_t)s.B * s.Hv * (s.Dv / kRows);
    return ctas * (nck_of(s) + kC) * kRows * (size_t)s.Dk * sizeof(float);
}

cudaError_t launch_backward(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const float *g, const float *beta, const float *state_in, const uint8_t *mask,
                            const uint16_t *dy, const float *dstate_out, float *dq, float *dk, float *dv,
                            float *dg, float *dbeta, float *dstate_in, void *ws, cudaStream_t st) {
    if (s.Dv % kRows != 0) return cudaErrorNotSupported;
    const size_t nqk = (size_t)s.B * s.T * s.Hk * s.Dk, nv = (size_t)s.B * s.T * s.Hv * s.Dv;
    const size_t ng = (size_t)s.B * s.T * s.Hv;
    cudaError_t e = cudaMemsetAsync(dq, 0, nqk * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dk, 0, nqk * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, nv * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dg, 0, ng * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dbeta, 0, ng * sizeof(float), st);
    if (e != cudaSuccess) return e;
    BwdParams p{q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk, dv, dg, dbeta, dstate_in,
                static_cast<float *>(ws), s.B, s.T, s.Hk, s.Hv, s.Dv, (int)nck_of(s)};
    switch (s.Dk) {
        case 32: return launch_bwd_t<32>(s, p, st);
        case 64: return launch_bwd_t<64>(s, p, st);
        case 128: return launch_bwd_t<128>(s, p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
