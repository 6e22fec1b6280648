// Sequential-form prefill: the gated delta rule run step by step with the
// state resident in registers for all T steps.
//
// Definition: "mlx-bun 0.4.0 -> 1.0.0, package/src/model/qwen3-delta.ts",
// gated_delta_step and its masked specialization (state rows per dv, decay,
// kv_mem, delta, update, output; a masked step writes y = 0 and skips the
// update); "mlex 0.1.2, src/models/gated_delta.rs", the per-timestep loop.
//
// A CTA (4 warps) owns R = 16*RPL rows of one (b, hv) state.  Lane (rg, cg) of
// warp w holds rows w*4*RPL + rg*RPL + i (i < RPL) and columns
// [cg*Dk/8, (cg+1)*Dk/8), so a row's dot products are shuffle sums over the 8
// lanes that share rg.  q/k/v tiles of 64 steps are staged in shared memory by
// 2-D TMA loads (double buffered, one mbarrier per stage); g, beta and the mask
// are gathered by plain loads one chunk ahead.  k.q per step is precomputed for
// the chunk so that y = g (S.q) + delta (k.q) needs no second reduction.
// Chunks whose 64 steps are all masked are skipped (zero y, no staging).
#include "common.cuh"
#include "internal.h"
#include "mask_scan.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;
constexpr int kTC = 64;   // steps per staged chunk

struct SeqParams {
    const float *g, *beta, *state_in;
    float *state_out;
    const uint8_t *mask;
    const int *order;   // row slot -> batch row (optional, with a mask)
    uint16_t *y;
    unsigned *err;
    int B, T, Hk, Hv, Dv;
};

__host__ __device__ constexpr int align128(int x) { return (x + 127) & ~127; }

template <int DK, int R, bool VEC>
struct SeqSmem {
    static constexpr int q_off = 0;
    static constexpr int k_off = q_off + align128(kTC * DK * 2);
    static constexpr int v_off = k_off + align128(kTC * DK * 2);
    static constexpr int g_off = v_off + align128(kTC * R * 2);
    static constexpr int b_off = g_off + kTC * 4;
    static constexpr int kq_off = b_off + kTC * 4;
    static constexpr int m_off = kq_off + kTC * 4;
    // per-channel gate tile [kTC][DK] f32 (vectorized gating only)
    static constexpr int gv_off = align128(m_off + kTC * 4);
    static constexpr int stage_bytes = VEC ? align128(gv_off + kTC * DK * 4) : align128(m_off + kTC * 4);
    static constexpr int y_off = 2 * stage_bytes;
    static constexpr int total = y_off + kTC * R * 4;
    static constexpr uint32_t tx_bytes = (uint32_t)(2 * kTC * DK * 2 + kTC * R * 2 + (VEC ? kTC * DK * 4 : 0));
};

template <int CW>
__device__ __forceinline__ void load_row_bf16(const uint16_t *p, float (&o)[CW]) {
    static_assert(CW % 4 == 0, "");
#pragma unroll
    for (int j = 0; j < CW; j += 4) {
        const uint2 r = *reinterpret_cast<const uint2 *>(p + j);
        o[j + 0] = __uint_as_float(r.x << 16);
        o[j + 1] = __uint_as_float(r.x & 0xffff0000u);
        o[j + 2] = __uint_as_float(r.y << 16);
        o[j + 3] = __uint_as_float(r.y & 0xffff0000u);
    }
}

// VEC: vectorized gating, one decay factor per key channel (g [B, T, Hv, Dk],
// staged by TMA with q/k/v); the state columns are decayed before the dots.
// MASKED: a step mask is given; wholly masked chunks are skipped.  (Without a
// mask the chunk loop is the plain one, compiled without the search.)
template <int DK, int RPL, bool VEC, bool MASKED>
__global__ void __launch_bounds__(kThreads) prefill_seq_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                               const __grid_constant__ CUtensorMap tm_k,
                                                               const __grid_constant__ CUtensorMap tm_v,
                                                               const __grid_constant__ CUtensorMap tm_g,
                                                               const SeqParams p) {
    constexpr int R = 16 * RPL;
    constexpr int CW = DK / 8;
    using L = SeqSmem<DK, R, VEC>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full_bar[2];
    __shared__ uint32_t scan_bits[ChunkScan<kThreads>::kWords];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = lane >> 3, cg = lane & 7;
    const int nslice = p.Dv / R;
    const int slice = blockIdx.x % nslice;
    const int hv = blockIdx.x / nslice;
    const int b = (MASKED && p.order != nullptr) ? p.order[blockIdx.y] : (int)blockIdx.y;
    const int G = p.Hv / p.Hk;
    const int hk = hv / G;
    const int r0 = slice * R;
    const int T = p.T;

    if (tid == 0) {
        mbar_init(&full_bar[0], 1);
        mbar_init(&full_bar[1], 1);
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }

    // state slice -> registers
    float s[RPL][CW];
    const size_t head_off = ((size_t)b * p.Hv + hv) * p.Dv;
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
        const int row = r0 + warp * 4 * RPL + rg * RPL + i;
        if (p.state_in != nullptr) {
            const float4 *src = reinterpret_cast<const float4 *>(p.state_in + (head_off + row) * DK + cg * CW);
#pragma unroll
            for (int j = 0; j < CW / 4; ++j) {
                const float4 x = src[j];
                s[i][4 * j] = x.x;
                s[i][4 * j + 1] = x.y;
                s[i][4 * j + 2] = x.z;
                s[i][4 * j + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < CW; ++j) s[i][j] = 0.0f;
        }
    }
    __syncthreads();

    const int nchunks = (T + kTC - 1) / kTC;
    auto issue = [&](int c, int st) {
        unsigned char *base = smem + st * L::stage_bytes;
        if (tid == 0) {
            mbar_expect_tx(&full_bar[st], L::tx_bytes);
            const int row = b * T + c * kTC;
            tma_load_2d(base + L::q_off, &tm_q, hk * DK, row, &full_bar[st]);
            tma_load_2d(base + L::k_off, &tm_k, hk * DK, row, &full_bar[st]);
            tma_load_2d(base + L::v_off, &tm_v, hv * p.Dv + r0, row, &full_bar[st]);
            if constexpr (VEC) tma_load_2d(base + L::gv_off, &tm_g, hv * DK, row, &full_bar[st]);
        }
        if (tid < kTC) {
            const int t = c * kTC + tid;
            float gg = 1.0f, bb = 0.0f;
            int m = 0;
            if (t < T) {
                const size_t gi = ((size_t)b * T + t) * p.Hv + hv;
                if constexpr (!VEC) gg = p.g[gi];
                bb = p.beta[gi];
                m = MASKED ? (p.mask[(size_t)b * T + t] != 0) : 1;
            }
            reinterpret_cast<float *>(base + L::g_off)[tid] = gg;
            reinterpret_cast<float *>(base + L::b_off)[tid] = bb;
            reinterpret_cast<int *>(base + L::m_off)[tid] = m;
        }
    };

    ChunkScan<kThreads> scan(MASKED ? p.mask + (size_t)b * T : nullptr, T, scan_bits);
    uint16_t *y_row0 = p.y + ((size_t)b * T * p.Hv + hv) * p.Dv + r0;
    const size_t y_stride = (size_t)p.Hv * p.Dv;
    int c = 0;
    if constexpr (MASKED) {
        c = scan.next_active(0);
        if (c > 0) zero_y_rows(y_row0, y_stride, 0, min(c * kTC, T), R);
    }
    if (c < nchunks) issue(c, 0);
    float *y_s = reinterpret_cast<float *>(smem + L::y_off);
    bool ok_all = true;

    // `it` counts the chunks actually processed: it picks the stage and the
    // stage barrier's phase
    for (int it = 0; c < nchunks; ++it) {
        const int st = it & 1;
        unsigned char *base = smem + st * L::stage_bytes;
        int cn = c + 1;
        if constexpr (MASKED) cn = scan.next_active(c + 1);
        if (cn < nchunks) issue(cn, st ^ 1);
        bool ok = mbar_wait(&full_bar[st], (uint32_t)((it >> 1) & 1), p.err);
        ok = __syncthreads_and(ok) != 0;
        if (!ok) {
            ok_all = false;
            break;
        }
        const uint16_t *qs = reinterpret_cast<const uint16_t *>(base + L::q_off);
        const uint16_t *ks = reinterpret_cast<const uint16_t *>(base + L::k_off);
        const uint16_t *vs = reinterpret_cast<const uint16_t *>(base + L::v_off);
        const float *gs = reinterpret_cast<const float *>(base + L::g_off);
        const float *bs = reinterpret_cast<const float *>(base + L::b_off);
        float *kqs = reinterpret_cast<float *>(base + L::kq_off);
        const int *ms = reinterpret_cast<const int *>(base + L::m_off);
        const int nt = min(kTC, T - c * kTC);

        // k.q per step of the chunk
        for (int t = warp; t < nt; t += kThreads / 32) {
            float acc = 0.0f;
            for (int j = lane; j < DK; j += 32)
                acc = fmaf(bf16_to_f32(ks[t * DK + j]), bf16_to_f32(qs[t * DK + j]), acc);
            acc = warp_sum(acc);
            if (lane == 0) kqs[t] = acc;
        }
        __syncthreads();

        for (int t = 0; t < nt; ++t) {
            if (ms[t] == 0) {
                if (cg == 0) {
#pragma unroll
                    for (int i = 0; i < RPL; ++i) y_s[t * R + warp * 4 * RPL + rg * RPL + i] = 0.0f;
                }
                continue;
            }
            float g = gs[t];
            const float beta = bs[t], kq = kqs[t];
            float kf[CW], qf[CW];
            load_row_bf16<CW>(ks + t * DK + cg * CW, kf);
            load_row_bf16<CW>(qs + t * DK + cg * CW, qf);
            if constexpr (VEC) {
                // decay each state column by its own factor, then proceed with g = 1
                const float *gt = reinterpret_cast<const float *>(base + L::gv_off) + t * DK + cg * CW;
#pragma unroll
                for (int j = 0; j < CW; j += 4) {
                    const float4 gv = *reinterpret_cast<const float4 *>(gt + j);
#pragma unroll
                    for (int i = 0; i < RPL; ++i) {
                        s[i][j] *= gv.x;
                        s[i][j + 1] *= gv.y;
                        s[i][j + 2] *= gv.z;
                        s[i][j + 3] *= gv.w;
                    }
                }
                g = 1.0f;
            }
            float dk[RPL], dq[RPL];
#pragma unroll
            for (int i = 0; i < RPL; ++i) {
                float a0 = 0.0f, a1 = 0.0f, b0 = 0.0f, b1 = 0.0f;
#pragma unroll
                for (int j = 0; j < CW; j += 2) {
                    a0 = fmaf(s[i][j], kf[j], a0);
                    a1 = fmaf(s[i][j + 1], kf[j + 1], a1);
                    b0 = fmaf(s[i][j], qf[j], b0);
                    b1 = fmaf(s[i][j + 1], qf[j + 1], b1);
                }
                dk[i] = a0 + a1;
                dq[i] = b0 + b1;
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
#pragma unroll
                for (int i = 0; i < RPL; ++i) {
                    dk[i] += __shfl_xor_sync(0xffffffffu, dk[i], o);
                    dq[i] += __shfl_xor_sync(0xffffffffu, dq[i], o);
                }
            }
#pragma unroll
            for (int i = 0; i < RPL; ++i) {
                const int rl = warp * 4 * RPL + rg * RPL + i;
                const float vv = bf16_to_f32(vs[t * R + rl]);
                const float delta = beta * (vv - g * dk[i]);
#pragma unroll
                for (int j = 0; j < CW; ++j) s[i][j] = fmaf(delta, kf[j], g * s[i][j]);
                if (cg == 0) y_s[t * R + rl] = fmaf(delta, kq, g * dq[i]);
            }
        }
        __syncthreads();

        // y tile -> global (bf16), R contiguous outputs per step
        for (int idx = tid; idx < nt * (R / 2); idx += kThreads) {
            const int t = idx / (R / 2), pr = idx % (R / 2);
            const uint32_t packed = (uint32_t)f32_to_bf16(y_s[t * R + 2 * pr]) |
                                    ((uint32_t)f32_to_bf16(y_s[t * R + 2 * pr + 1]) << 16);
            uint16_t *dst = p.y + (((size_t)b * T + c * kTC + t) * p.Hv + hv) * p.Dv + r0 + 2 * pr;
            *reinterpret_cast<uint32_t *>(dst) = packed;
        }
        if constexpr (MASKED) {
            if (cn > c + 1) zero_y_rows(y_row0, y_stride, min((c + 1) * kTC, T), min(cn * kTC, T), R);
        }
        c = cn;
    }

    if (!ok_all) return;
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
        const int row = r0 + warp * 4 * RPL + rg * RPL + i;
        float4 *dst = reinterpret_cast<float4 *>(p.state_out + (head_off + row) * DK + cg * CW);
#pragma unroll
        for (int j = 0; j < CW / 4; ++j)
            dst[j] = make_float4(s[i][4 * j], s[i][4 * j + 1], s[i][4 * j + 2], s[i][4 * j + 3]);
    }
}

template <int DK, int RPL, bool VEC, bool MASKED>
cudaError_t launch_seq_m(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const SeqParams &p, cudaStream_t st) {
    constexpr int R = 16 * RPL;
    using L = SeqSmem<DK, R, VEC>;
    CUtensorMap tq, tk, tv, tg;
    const uint64_t rows = (uint64_t)s.B * (uint64_t)(s.T > 0 ? s.T : 1);
    if (!encode_tmap_2d(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, (uint64_t)s.Hk * DK, kTC, DK) ||
        !encode_tmap_2d(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, (uint64_t)s.Hk * DK, kTC, DK) ||
        !encode_tmap_2d(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, (uint64_t)s.Hv * s.Dv, kTC, R))
        return cudaErrorInvalidValue;
    if constexpr (VEC) {
        if (!encode_tmap_2d(&tg, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, rows, (uint64_t)s.Hv * DK, kTC, DK))
            return cudaErrorInvalidValue;
    } else {
        tg = tq;   // unused
    }
    static unsigned long long attr_done = 0;   // per instantiation, one bit per device
    cudaError_t ae = set_max_smem(attr_done, prefill_seq_kernel<DK, RPL, VEC, MASKED>, (size_t)L::total);
    if (ae != cudaSuccess) return ae;
    dim3 grid(s.Hv * (s.Dv / R), s.B);
    prefill_seq_kernel<DK, RPL, VEC, MASKED><<<grid, kThreads, L::total, st>>>(tq, tk, tv, tg, p);
    return cudaGetLastError();
}

template <int DK, int RPL, bool VEC>
cudaError_t launch_seq_t(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const SeqParams &p, cudaStream_t st) {
    return p.mask != nullptr ? launch_seq_m<DK, RPL, VEC, true>(s, q, k, v, p, st)
                             : launch_seq_m<DK, RPL, VEC, false>(s, q, k, v, p, st);
}

template <bool VEC>
cudaError_t launch_seq_any(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const SeqParams &p, cudaStream_t st) {
    // 32-row CTAs when there are enough of them to fill the GPU, else 16-row
    const long ctas32 = (long)s.B * s.Hv * (s.Dv / 32);
    const bool small = ctas32 < num_sms();
    switch (s.Dk) {
        case 32:
            return small ? launch_seq_t<32, 1, VEC>(s, q, k, v, p, st) : launch_seq_t<32, 2, VEC>(s, q, k, v, p, st);
        case 64:
            return small ? launch_seq_t<64, 1, VEC>(s, q, k, v, p, st) : launch_seq_t<64, 2, VEC>(s, q, k, v, p, st);
        case 128:
            return small ? launch_seq_t<128, 1, VEC>(s, q, k, v, p, st)
                         : launch_seq_t<128, 2, VEC>(s, q, k, v, p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prefill_seq(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const float *g, const float *beta, const float *state_in, float *state_out,
                               const uint8_t *mask, const int *order, uint16_t *y, unsigned *err,
                               cudaStream_t st) {
    SeqParams p{g, beta, state_in, state_out, mask, order, y, err, s.B, s.T, s.Hk, s.Hv, s.Dv};
    return launch_seq_any<false>(s, q, k, v, p, st);
}

cudaError_t launch_prefill_seq_vec(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                   const float *g_vec, const float *beta, const float *state_in, float *state_out,
                                   const uint8_t *mask, uint16_t *y, unsigned *err, cudaStream_t st) {
    SeqParams p{g_vec, beta, state_in, state_out, mask, nullptr, y, err, s.B, s.T, s.Hk, s.Hv, s.Dv};
    return launch_seq_any<true>(s, q, k, v, p, st);
}

}  // namespace gdn
