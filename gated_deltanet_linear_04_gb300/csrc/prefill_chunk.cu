// Chunked (WY / UT-transform) prefill on the 5th-generation tensor cores.
//
// The recurrence of "mlex 0.1.2, src/models/gated_delta.rs" (GatedDeltaNet::
// forward, per-timestep loop) and of the gated_delta_step kernel of "mlx-bun
// 0.4.0 -> 1.0.0, package/src/model/qwen3-delta.ts" is re-blocked exactly into
// chunks of 64 steps.  For a chunk with start state S0 ([Dv, Dk]) and
// log-decay prefix sums lg_r = sum_{i<=r} log g_i (held in base 2 below):
//   A[r,i] = beta_r exp(lg_r - lg_i) (k_r . k_i), i < r;   T = (I + A)^-1
//   U = T diag(beta) V,   W = T diag(beta exp(lg)) K,   D = U - W S0^T
//   Y = diag(exp(lg)) Q S0^T + (M o Q K^T) D,   M[r,i] = exp(lg_r - lg_i), i <= r
//   S = exp(lg_63) S0 + D^T diag(exp(lg_63 - lg)) K
// (A masked step enters with g = 1, beta = 0; its y is written as zero.)
//
// Every product is issued in transposed form so that the MMA row count is
// M = 128 (= Dv or Dk) and the accumulator row is one TMEM lane:
//   [K;Q] K^T        bf16 x bf16  -> TMEM QK   (rows 0-63 K K^T, 64-127 Q K^T)
//   U^T = (bV)^T T^T tf32         -> TMEM D
//   W^T = (bgK)^T T^T tf32        -> TMEM W
//   D^T += S0 (-W)^T tf32         -> TMEM D    (accumulates onto U^T)
//   Y^T = S0 (gQ)^T  tf32         -> TMEM Y
//   Y^T += D^T P^T   tf32         -> TMEM Y
//   S  += D^T Kc^T   tf32         -> TMEM S    (S pre-scaled by exp(lg_63))
// The f32 state lives in TMEM across all chunks and accumulates in f32; the D
// and Y products read it straight from TMEM as their A operand (the tensor
// core takes the top 19 bits, i.e. tf32 by truncation).  The 64 x 64 unit
// lower-triangular inverse T is computed on the CUDA cores by blocked doubling
// (8x8 diagonal blocks, then 16-, 32-, 64-wide merges X = -T_bb A_ba T_aa).
// q, k, v tiles arrive by 2-D TMA (k and q 128B-swizzled straight into the
// MMA operand layout), prefetched one chunk ahead.
//
// One CTA (256 threads) owns one (b, hv) head for all T.  Supports Dk = Dv =
// 128.  Shared memory: 13 slots of 16 KiB reused across the phases of a chunk.
// Chunks whose 64 steps are all masked are skipped: their y is written zero and
// their inputs are never staged.
//
// NORM variant: each chunk's output is the layer's RMSNormGated of y ("mlex
// 0.1.2, src/models/gated_delta.rs", GatedDeltaNet::forward: f32 rms_norm of
// the bf16 y over Dv, times the norm weight, times silu(z), cast to bf16),
// computed from the bf16 y staging tile with the z tile brought in by TMA,
// so y itself never goes to memory.
#include "common.cuh"
#include "internal.h"
#include "mask_scan.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kC = 64;          // chunk length
constexpr int kD = 128;         // Dk = Dv
constexpr uint32_t kSlot = 16384;
constexpr int kSlots = 13;
constexpr uint32_t kSmemBytes = kSlots * kSlot + 1024;

// slot map (byte offsets from the 1024-aligned base)
constexpr uint32_t S_KQ = 0 * kSlot;    // 2 slots: K rows 0-63 / Q rows 64-127, K-halves of 64
constexpr uint32_t S_V = 2 * kSlot;     // plain [64][128] bf16
constexpr uint32_t S_GQ = 3 * kSlot;    // 2 slots: (g Q) [64][128] tf32, 4 K-tiles of 8 KiB
constexpr uint32_t S_KT = 5 * kSlot;    // 2 slots: Kc^T [128][64] tf32, 2 K-tiles of 16 KiB
constexpr uint32_t S_BV = 7 * kSlot;    // 2 slots: (b V)^T [128][64]  -> later D^T
constexpr uint32_t S_BK = 9 * kSlot;    // 2 slots: (b g K)^T [128][64] -> later y staging
constexpr uint32_t S_A = 11 * kSlot;    // A / T plain [64][64] f32     -> later (-W) tiles 0,1 -> P
constexpr uint32_t S_T = 12 * kSlot;    // Y scratch, then T [64][64] tf32 -> later (-W) tiles 2,3
constexpr uint32_t S_NW = S_A;          // -W [64][128] tf32, 4 K-tiles of 8 KiB (slots 11-12)
constexpr uint32_t S_DT = S_BV;         // D^T [128][64] tf32, 2 K-tiles of 16 KiB (slots 7-8)
constexpr uint32_t S_P = S_A;           // P [64][64] tf32, 2 K-tiles of 8 KiB (slot 11)
constexpr uint32_t S_YST = S_BK;        // y staging [64][128] bf16 (slot 9, free after the W product)
constexpr uint32_t S_Z = S_GQ;          // NORM: z tile [64][128] bf16 (slot 3, free after the S0 products)

// TMEM columns
constexpr uint32_t C_QK = 0, C_D = 64, C_W = 128, C_Y = 192, C_S = 256, kTmemCols = 512;

struct ChunkParams {
    const float *g, *beta, *state_in;
    float *state_out;
    const uint8_t *mask;
    const int *order;   // row slot -> batch row (optional, with a mask)
    uint16_t *y;        // y, or the gated-norm output for the NORM variant
    const float *norm_w;
    float norm_eps;
    unsigned *err;
    int B, T, Hk, Hv;
};

// A / T working matrix, row-major; groups of 4 columns are XOR-permuted by the
// row (r % 8) so that row-per-thread float4 stores spread over all banks while
// each aligned group of 4 stays contiguous for float4 loads.
__device__ __forceinline__ int aidx(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

// Log-decay prefix sums are kept in base 2 (lg_r = sum_{i<=r} log2 g_i).
// 2^x of a non-positive difference with the hardware base-2 exponential
// (ex2.approx: relative error ~2^-22, far below the tf32 rounding these
// factors go through; results below 2^-126 flush to zero, which is the limit
// the decay takes anyway).  The precise library exp2f path measured ~3x slower
// for the 64 x 64 ratio matrices built every chunk.
__device__ __forceinline__ float decay(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// log2 of a gate value with the hardware base-2 logarithm (lg2.approx, not
// flushing subnormal inputs), clamped at -250: a gate of exactly 0 (or one
// that underflowed) then decays everything before it to 2^-250, which is 0
// in f32, instead of making the prefix sums -inf and their differences NaN.
// A gate of exactly 1 (every masked step) gives exactly 0.
__device__ __forceinline__ float log2_gate(float g) {
    float r;
    asm("lg2.approx.f32 %0, %1;" : "=f"(r) : "f"(g));
    return g == 1.0f ? 0.0f : fmaxf(r, -250.0f);
}

// One merge level of the blocked inverse: for each pair of S x S diagonal
// blocks (a = [q0, q0+S), b = [q0+S, q0+2S)) of the unit lower triangular
// T = (I + A)^-1, the lower-left block is X = -T_bb A_ba T_aa.  Each task
// computes 4 adjacent columns of one row; sums run over full blocks because
// the triangular factors hold explicit zeros above the diagonal.
template <int S>
__device__ __forceinline__ void merge_level(float *As, float *Ys, int tid) {
    constexpr int G4 = S / 4;
    constexpr int NT = (32 / S) * S * G4;
    const int pi = tid / (S * G4), rem = tid % (S * G4), r = rem / G4, c = (rem % G4) * 4, q0 = pi * 2 * S;
    if (tid < NT) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m < S; ++m) {
            const float a = As[aidx(q0 + S + r, q0 + m)];
            const float4 t = ld4(As + aidx(q0 + m, q0 + c));
            acc.x = fmaf(a, t.x, acc.x);
            acc.y = fmaf(a, t.y, acc.y);
            acc.z = fmaf(a, t.z, acc.z);
            acc.w = fmaf(a, t.w, acc.w);
        }
        st4(Ys + (pi * S + r) * S + c, acc);
    }
    __syncthreads();
    if (tid < NT) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m < S; ++m) {
            const float t = As[aidx(q0 + S + r, q0 + S + m)];
            const float4 yv = ld4(Ys + (pi * S + m) * S + c);
            acc.x = fmaf(t, yv.x, acc.x);
            acc.y = fmaf(t, yv.y, acc.y);
            acc.z = fmaf(t, yv.z, acc.z);
            acc.w = fmaf(t, yv.w, acc.w);
        }
        st4(As + aidx(q0 + S + r, q0 + c), make_float4(-acc.x, -acc.y, -acc.z, -acc.w));
    }
    __syncthreads();
}

__device__ __forceinline__ void st_tf32x4(uint8_t *base, uint32_t off, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(base + off) =
        make_float4(umma::to_tf32(a), umma::to_tf32(b), umma::to_tf32(c), umma::to_tf32(d));
}

__device__ __forceinline__ float kq_elem(const uint8_t *sm, int row, int dk) {
    // row 0-63: K, 64-127: Q; bf16, 128B swizzle, K-halves of 64 in two slots
    const uint16_t *p = reinterpret_cast<const uint16_t *>(
        sm + S_KQ + (dk >> 6) * kSlot + umma::sw128((uint32_t)row, (uint32_t)(dk & 63) * 2));
    return bf16_to_f32(*p);
}

template <bool NORM>
__global__ void __launch_bounds__(kThreads, 1) prefill_chunk_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                     const __grid_constant__ CUtensorMap tm_q,
                                                                     const __grid_constant__ CUtensorMap tm_v,
                                                                     const __grid_constant__ CUtensorMap tm_z,
                                                                     const ChunkParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_tma, bar_mma, bar_z;
    __shared__ float s_w[NORM ? kD : 1];
    __shared__ uint32_t tmem_slot;
    __shared__ float s_g[2][kC], s_b[2][kC];
    __shared__ int s_m[2][kC];
    __shared__ __align__(16) float s_lg[kC];
    __shared__ __align__(16) float s_gam[kC];
    __shared__ __align__(16) float s_beta[kC];
    __shared__ __align__(16) float s_bg[kC];
    __shared__ __align__(16) float s_kc[kC];
    __shared__ uint32_t scan_bits[ChunkScan<kThreads>::kWords];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3;                 // TMEM lane quarter of this warp
    const int half = warp >> 2;                // which half of the columns this warp handles
    const int row = quad * 32 + lane;          // TMEM lane / accumulator row of this thread
    const int hv = blockIdx.x;
    const int b = p.order != nullptr ? p.order[blockIdx.y] : (int)blockIdx.y;
    const int hk = hv / (p.Hv / p.Hk);
    const int T = p.T;
    const int nchunks = (T + kC - 1) / kC;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - smem_u32(smem_raw));
    float *As = reinterpret_cast<float *>(sm + S_A);
    float *Ys = reinterpret_cast<float *>(sm + S_T);

    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_z, 1);
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_v);
        if constexpr (NORM) prefetch_tmap(&tm_z);
    }
    if constexpr (NORM) {
        for (int i = tid; i < kD; i += kThreads) s_w[i] = p.norm_w[i];
    }
    if (warp == 0) {
        umma::tmem_alloc(&tmem_slot, kTmemCols);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;

    // ---- initial state -> TMEM S (row = dv, columns = dk); half 0: dk 0-63, half 1: 64-127
    {
        const size_t off = (((size_t)b * p.Hv + hv) * kD + row) * kD + half * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float r[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (p.state_in != nullptr) x = *reinterpret_cast<const float4 *>(p.state_in + off + c * 32 + j);
                r[j] = x.x; r[j + 1] = x.y; r[j + 2] = x.z; r[j + 3] = x.w;
            }
            umma::tmem_st32(tmem + lane_base + C_S + half * 64 + c * 32, r);
        }
        umma::tmem_st_wait();
    }

    // per-step g, beta, mask of a chunk: gathered into registers early (threads
    // < 64, one step each) and published to shared memory later, so the global
    // load latency never sits in front of a block barrier
    float pf_g = 1.0f, pf_b = 0.0f;
    int pf_m = 0;
    auto gather_steps = [&](int c) {
        pf_g = 1.0f;
        pf_b = 0.0f;
        pf_m = 0;
        const int t = c * kC + tid;
        if (tid < kC && t < T) {
            const size_t gi = ((size_t)b * T + t) * p.Hv + hv;
            pf_m = p.mask == nullptr ? 1 : (p.mask[(size_t)b * T + t] != 0);
            if (pf_m) {
                pf_g = p.g[gi];
                pf_b = p.beta[gi];
            }
        }
    };
    auto publish_steps = [&](int slot) {
        if (tid < kC) {
            s_g[slot][tid] = pf_g;
            s_b[slot][tid] = pf_b;
            s_m[slot][tid] = pf_m;
        }
    };
    auto issue_tma = [&](int c) {
        if (tid == 0) {
            mbar_expect_tx(&bar_tma, 4 * 8192 + 16384);
            const int rowg = b * T + c * kC;
            tma_load_2d(sm + S_KQ, &tm_k, hk * kD, rowg, &bar_tma);
            tma_load_2d(sm + S_KQ + kSlot, &tm_k, hk * kD + 64, rowg, &bar_tma);
            tma_load_2d(sm + S_KQ + 8192, &tm_q, hk * kD, rowg, &bar_tma);
            tma_load_2d(sm + S_KQ + kSlot + 8192, &tm_q, hk * kD + 64, rowg, &bar_tma);
            tma_load_2d(sm + S_V, &tm_v, hv * kD, rowg, &bar_tma);
        }
    };

    uint32_t mma_phase = 0;
    bool ok = true;
    bool z_pending = false;     // thread 0: a z copy was issued and not yet waited on
    uint32_t z_parity = 0;
    // bounded wait on the MMA barrier by every thread, agreed across the CTA
    auto wait_mma = [&]() {
        bool w = mbar_wait(&bar_mma, mma_phase & 1u, p.err);
        ++mma_phase;
        w = __syncthreads_and(w) != 0;
        umma::fence_after_sync();
        return w;
    };
    // make generic smem writes and TMEM stores visible to the next MMA issue
    auto publish = [&]() {
        fence_proxy_async_smem();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
    };

    ChunkScan<kThreads> scan(p.mask == nullptr ? nullptr : p.mask + (size_t)b * T, T, scan_bits);
    uint16_t *y_row0 = p.y + (size_t)b * T * p.Hv * kD + (size_t)hv * kD;
    const size_t y_stride = (size_t)p.Hv * kD;
    int c = scan.next_active(0);
    zero_y_rows(y_row0, y_stride, 0, min(c * kC, T), kD);
    if (c < nchunks) {
        issue_tma(c);
        gather_steps(c);
        publish_steps(0);
    }
    __syncthreads();

    // `it` counts the chunks actually processed: it picks the step-slot and
    // the TMA barrier's phase
    for (int it = 0; c < nchunks && ok; ++it) {
        const int st = it & 1;
        const int t0 = c * kC;
        // ---- S1: chunk inputs, log-decay prefix sums (warp 0)
        ok = mbar_wait(&bar_tma, (uint32_t)(it & 1), p.err);
        if (warp == 0) {
            const float la = log2_gate(s_g[st][2 * lane]), lb = log2_gate(s_g[st][2 * lane + 1]);
            float incl = la + lb;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            const float up = __shfl_up_sync(0xffffffffu, incl, 1);
            const float excl = lane == 0 ? 0.0f : up;
            const float lg0 = excl + la, lg1 = lg0 + lb;
            const float last = __shfl_sync(0xffffffffu, incl, 31);
            s_lg[2 * lane] = lg0;
            s_lg[2 * lane + 1] = lg1;
            const float e0 = decay(lg0), e1 = decay(lg1);
            s_gam[2 * lane] = e0;
            s_gam[2 * lane + 1] = e1;
            s_kc[2 * lane] = decay(last - lg0);
            s_kc[2 * lane + 1] = decay(last - lg1);
            const float b0 = s_b[st][2 * lane], b1 = s_b[st][2 * lane + 1];
            s_beta[2 * lane] = b0;
            s_beta[2 * lane + 1] = b1;
            s_bg[2 * lane] = b0 * e0;
            s_bg[2 * lane + 1] = b1 * e1;
        }
        ok = __syncthreads_and(ok) != 0;
        if (!ok) break;

        const int cn = scan.next_active(c + 1);
        if (cn < nchunks) gather_steps(cn);
        // ---- S2: [K;Q] K^T on the tensor core; meanwhile build the tf32 operands
        if (tid == 0) {
            umma::fence_after_sync();
            const uint32_t id = umma::idesc(128, 64, umma::kFmtBF16);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t a = base + S_KQ + (k >> 2) * kSlot + (k & 3) * 32;
                umma::mma_bf16(tmem + C_QK, umma::desc_sw128(a), umma::desc_sw128(a), id, k > 0);
            }
            umma::mma_commit(&bar_mma);
        }
        // (g Q)[r][dk]: a warp covers one row r, 4 consecutive dk per lane
        for (int i = tid; i < kC * kD / 4; i += kThreads) {
            const int r = i >> 5, dk = (i & 31) * 4;
            const float gm = s_gam[r];
            const uint2 qq = *reinterpret_cast<const uint2 *>(
                sm + S_KQ + (dk >> 6) * kSlot + umma::sw128(64 + r, (dk & 63) * 2));
            st_tf32x4(sm, S_GQ + (dk >> 5) * 8192 + umma::sw128(r, (dk & 31) * 4),
                      gm * __uint_as_float(qq.x << 16), gm * __uint_as_float(qq.x & 0xffff0000u),
                      gm * __uint_as_float(qq.y << 16), gm * __uint_as_float(qq.y & 0xffff0000u));
        }
        // Kc^T[dk][r] and (b g K)^T[dk][r]: lanes take consecutive dk (conflict-free
        // reads along a K row), each thread 4 consecutive r
        for (int i = tid; i < kD * kC / 4; i += kThreads) {
            const int dk = i & (kD - 1), r = (i >> 7) * 4;
            const float k0 = kq_elem(sm, r, dk), k1 = kq_elem(sm, r + 1, dk), k2 = kq_elem(sm, r + 2, dk),
                        k3 = kq_elem(sm, r + 3, dk);
            const uint32_t off = (r >> 5) * kSlot + umma::sw128(dk, (r & 31) * 4);
            const float4 kc = ld4(s_kc + r), bg = ld4(s_bg + r);
            st_tf32x4(sm, S_KT + off, kc.x * k0, kc.y * k1, kc.z * k2, kc.w * k3);
            st_tf32x4(sm, S_BK + off, bg.x * k0, bg.y * k1, bg.z * k2, bg.w * k3);
        }
        // (b V)^T[dv][i]
        {
            const uint16_t *Vs = reinterpret_cast<const uint16_t *>(sm + S_V);
            for (int i = tid; i < kD * kC / 4; i += kThreads) {
                const int dv = i & (kD - 1), r = (i >> 7) * 4;
                const float4 be = ld4(s_beta + r);
                st_tf32x4(sm, S_BV + (r >> 5) * kSlot + umma::sw128(dv, (r & 31) * 4),
                          be.x * bf16_to_f32(Vs[r * kD + dv]), be.y * bf16_to_f32(Vs[(r + 1) * kD + dv]),
                          be.z * bf16_to_f32(Vs[(r + 2) * kD + dv]), be.w * bf16_to_f32(Vs[(r + 3) * kD + dv]));
            }
        }

        // ---- S3: A from K K^T (lanes 0-63)
        if (!wait_mma()) { ok = false; break; }
        if (quad < 2) {
            float kk[32];
            umma::tmem_ld32(tmem + lane_base + C_QK + half * 32, kk);
            umma::tmem_ld_wait();
            const int r = row;                      // 0..63
            const float lr = s_lg[r], br = s_beta[r];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const int i = half * 32 + j;
                const float4 li = ld4(s_lg + i);
                float4 v;
                v.x = i < r ? br * decay(lr - li.x) * kk[j] : 0.0f;
                v.y = i + 1 < r ? br * decay(lr - li.y) * kk[j + 1] : 0.0f;
                v.z = i + 2 < r ? br * decay(lr - li.z) * kk[j + 2] : 0.0f;
                v.w = i + 3 < r ? br * decay(lr - li.w) * kk[j + 3] : 0.0f;
                st4(As + aidx(r, i), v);
            }
        }
        // K and V tiles are no longer read: prefetch the next chunk
        umma::fence_before_sync();
        __syncthreads();
        if (cn < nchunks) {
            issue_tma(cn);
            publish_steps(st ^ 1);
        }

        // ---- S4: T = (I + A)^-1 by blocked doubling, in place in As
        {
            // 8 x 8 diagonal blocks by forward substitution: thread (block, column j)
            const int o = (tid >> 3) * 8, j = tid & 7;
            float t[8];
            if (tid < 64) {
                float a[8][8];
#pragma unroll
                for (int r = 1; r < 8; ++r)
#pragma unroll
                    for (int i = 0; i < r; ++i) a[r][i] = As[aidx(o + r, o + i)];
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    float acc = r == j ? 1.0f : 0.0f;
#pragma unroll
                    for (int i = 0; i < r; ++i) acc = fmaf(-a[r][i], t[i], acc);
                    t[r] = acc;
                }
            }
            __syncthreads();
            if (tid < 64) {
#pragma unroll
                for (int r = 0; r < 8; ++r) As[aidx(o + r, o + j)] = t[r];
            }
            __syncthreads();
        }
        merge_level<8>(As, Ys, tid);
        merge_level<16>(As, Ys, tid);
        merge_level<32>(As, Ys, tid);
        // T -> tf32 B operand [r][i] (slot S_T; the Y scratch is dead)
        for (int i = tid; i < kC * kC / 4; i += kThreads) {
            const int r = i >> 4, c4 = (i & 15) * 4;
            const float4 tv = ld4(As + aidx(r, c4));
            st_tf32x4(sm, S_T + (c4 >> 5) * 8192 + umma::sw128(r, (c4 & 31) * 4), tv.x, tv.y, tv.z, tv.w);
        }
        publish();

        // ---- S5: U^T and W^T on the tensor core
        if (tid == 0) {
            const uint32_t id = umma::idesc(128, 64, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t kt = k >> 2, ko = (k & 3) * 32;
                const uint64_t bt = umma::desc_sw128(base + S_T + kt * 8192 + ko);
                umma::mma_tf32(tmem + C_D, umma::desc_sw128(base + S_BV + kt * kSlot + ko), bt, id, k > 0);
                umma::mma_tf32(tmem + C_W, umma::desc_sw128(base + S_BK + kt * kSlot + ko), bt, id, k > 0);
            }
            umma::mma_commit(&bar_mma);
        }
        if (!wait_mma()) { ok = false; break; }
        // -W -> smem (B operand of the D update)
        {
            float wv[32];
            umma::tmem_ld32(tmem + lane_base + C_W + half * 32, wv);
            umma::tmem_ld_wait();
            const int dk = row;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = half * 32 + j;
                *reinterpret_cast<float *>(sm + S_NW + (dk >> 5) * 8192 + umma::sw128(r, (dk & 31) * 4)) =
                    umma::to_tf32(-wv[j]);
            }
        }
        publish();

        // ---- S6: D^T += S0 (-W)^T ; Y^T = S0 (gQ)^T
        if (tid == 0) {
            const uint32_t id = umma::idesc(128, 64, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                // A = the f32 state itself, read from TMEM (used as tf32)
                const uint32_t kt = k >> 2, ko = (k & 3) * 32, a = tmem + C_S + 8 * k;
                umma::mma_tf32_tmem_a(tmem + C_D, a, umma::desc_sw128(base + S_NW + kt * 8192 + ko), id, true);
                umma::mma_tf32_tmem_a(tmem + C_Y, a, umma::desc_sw128(base + S_GQ + kt * 8192 + ko), id, k > 0);
            }
            umma::mma_commit(&bar_mma);
        }
        if (!wait_mma()) { ok = false; break; }

        // ---- S7: D^T -> smem (A operand); P = M o Q K^T -> smem (B operand);
        // S <- exp(lg_63) S in TMEM (the D and Y products have read S already)
        if constexpr (NORM) {
            // the gQ slot is free now: bring in this chunk's z tile
            if (tid == 0) {
                mbar_expect_tx(&bar_z, 16384);
                tma_load_2d(sm + S_Z, &tm_z, hv * kD, b * T + t0, &bar_z);
                z_pending = true;
                z_parity = (uint32_t)(it & 1);
            }
        }
        {
            const float gl = s_gam[kC - 1];
#pragma unroll
            for (int cpart = 0; cpart < 2; ++cpart) {
                float sv[32];
                const uint32_t col = C_S + half * 64 + cpart * 32;
                umma::tmem_ld32(tmem + lane_base + col, sv);
                umma::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) sv[j] *= gl;
                umma::tmem_st32(tmem + lane_base + col, sv);
            }
        }
        {
            // both TMEM reads in flight before the one wait
            float dv[32], qk[32];
            umma::tmem_ld32(tmem + lane_base + C_D + half * 32, dv);
            if (quad >= 2) umma::tmem_ld32(tmem + lane_base + C_QK + half * 32, qk);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                st_tf32x4(sm, S_DT + half * kSlot + umma::sw128(row, j * 4), dv[j], dv[j + 1], dv[j + 2], dv[j + 3]);
            if (quad >= 2) {
                const int r = row - 64;
                const float lr = s_lg[r];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float v4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = half * 32 + j + e;
                        v4[e] = i <= r ? decay(lr - s_lg[i]) * qk[j + e] : 0.0f;
                    }
                    st_tf32x4(sm, S_P + half * 8192 + umma::sw128(r, j * 4), v4[0], v4[1], v4[2], v4[3]);
                }
            }
        }
        publish();

        // ---- S8: Y^T += D^T P^T ; S += D^T Kc^T
        if (tid == 0) {
            const uint32_t idy = umma::idesc(128, 64, umma::kFmtTF32);
            const uint32_t ids = umma::idesc(128, 128, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t kt = k >> 2, ko = (k & 3) * 32;
                const uint64_t a = umma::desc_sw128(base + S_DT + kt * kSlot + ko);
                umma::mma_tf32(tmem + C_Y, a, umma::desc_sw128(base + S_P + kt * 8192 + ko), idy, true);
                umma::mma_tf32(tmem + C_S, a, umma::desc_sw128(base + S_KT + kt * kSlot + ko), ids, true);
            }
            umma::mma_commit(&bar_mma);
        }
        if (!wait_mma()) { ok = false; break; }

        // ---- S9: y through a shared staging tile [64 steps][128 dv] bf16, then
        // 16-byte stores of the valid steps (masked steps are zero)
        {
            float yv[32];
            umma::tmem_ld32(tmem + lane_base + C_Y + half * 32, yv);
            umma::tmem_ld_wait();
            uint16_t *Yst = reinterpret_cast<uint16_t *>(sm + S_YST);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = half * 32 + j;
                Yst[r * kD + row] = s_m[st][r] ? f32_to_bf16(yv[j]) : (uint16_t)0;
            }
        }
        umma::fence_before_sync();
        __syncthreads();
        if constexpr (NORM) {
            // gated RMS norm per step: 4 threads per step, each covering the
            // 16-byte column groups qd, qd + 4, qd + 8, qd + 12 of the row
            if (!mbar_wait(&bar_z, (uint32_t)(it & 1), p.err)) ok = false;
            z_pending = false;
            const int r = tid >> 2, qd = tid & 3;
            uint8_t *yrow = sm + S_YST + r * kD * 2;
            const uint8_t *zrow = sm + S_Z + r * kD * 2;
            float ss = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 u = *reinterpret_cast<const uint4 *>(yrow + (j * 4 + qd) * 16);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
                    ss = fmaf(lo, lo, ss);
                    ss = fmaf(hi, hi, ss);
                }
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            const float rs = 1.0f / sqrtf(ss * (1.0f / (float)kD) + p.norm_eps);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c16 = j * 4 + qd;
                const uint4 u = *reinterpret_cast<const uint4 *>(yrow + c16 * 16);
                const uint4 zz = *reinterpret_cast<const uint4 *>(zrow + c16 * 16);
                const uint32_t yw[4] = {u.x, u.y, u.z, u.w}, zw[4] = {zz.x, zz.y, zz.z, zz.w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int dv = c16 * 8 + 2 * e;
                    const float y0 = __uint_as_float(yw[e] << 16), y1 = __uint_as_float(yw[e] & 0xffff0000u);
                    const float z0 = __uint_as_float(zw[e] << 16), z1 = __uint_as_float(zw[e] & 0xffff0000u);
                    const float o0 = silu(z0) * ((y0 * rs) * s_w[dv]);
                    const float o1 = silu(z1) * ((y1 * rs) * s_w[dv + 1]);
                    o[e] = (uint32_t)f32_to_bf16(o0) | ((uint32_t)f32_to_bf16(o1) << 16);
                }
                *reinterpret_cast<uint4 *>(yrow + c16 * 16) = make_uint4(o[0], o[1], o[2], o[3]);
            }
            ok = __syncthreads_and(ok) != 0;
            if (!ok) break;
        }
        {
            const int nv = min(kC, T - t0);
            for (int i = tid; i < nv * (kD / 8); i += kThreads) {
                const int r = i / (kD / 8), c8 = (i % (kD / 8)) * 8;
                *reinterpret_cast<uint4 *>(p.y + (((size_t)b * T + t0 + r) * p.Hv + hv) * kD + c8) =
                    *reinterpret_cast<const uint4 *>(sm + S_YST + (r * kD + c8) * 2);
            }
        }
        zero_y_rows(y_row0, y_stride, min((c + 1) * kC, T), min(cn * kC, T), kD);
        c = cn;
    }

    // ---- final state (only when every wait succeeded)
    if (__syncthreads_and(ok)) {
        const size_t off = (((size_t)b * p.Hv + hv) * kD + row) * kD + half * 64;
#pragma unroll
        for (int cpart = 0; cpart < 2; ++cpart) {
            float sv[32];
            umma::tmem_ld32(tmem + lane_base + C_S + half * 64 + cpart * 32, sv);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(p.state_out + off + cpart * 32 + j) =
                    make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
        }
    } else if (tid == 0) {
        // a wait gave up: give in-flight MMAs (and a z copy) a bounded chance to drain
        mbar_wait(&bar_mma, mma_phase & 1u, nullptr);
        if (z_pending) mbar_wait(&bar_z, z_parity, nullptr);
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

template <bool NORM>
cudaError_t set_smem_attr() {
    static bool attr_set = false;   // per instantiation; benign race
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_chunk_kernel<NORM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_prefill_chunked(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                   const float *g, const float *beta, const float *state_in, float *state_out,
                                   const uint8_t *mask, const int *order, uint16_t *y, const uint16_t *z,
                                   const float *norm_w, float norm_eps, unsigned *err, cudaStream_t st) {
    if (s.Dk != kD || s.Dv != kD) return cudaErrorNotSupported;
    CUtensorMap tk, tq, tv, tz;
    const uint64_t rows = (uint64_t)s.B * (uint64_t)s.T;
    if (!encode_tmap_2d(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, (uint64_t)s.Hk * kD, kC, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, (uint64_t)s.Hk * kD, kC, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, (uint64_t)s.Hv * kD, kC, kD,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    tz = tv;   // unused without the norm
    if (z != nullptr && !encode_tmap_2d(&tz, z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, (uint64_t)s.Hv * kD, kC,
                                        kD, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    cudaError_t e = z != nullptr ? set_smem_attr<true>() : set_smem_attr<false>();
    if (e != cudaSuccess) return e;
    ChunkParams p{g, beta, state_in, state_out, mask, mask != nullptr ? order : nullptr, y, norm_w, norm_eps, err,
                  s.B, s.T, s.Hk, s.Hv};
    dim3 grid(s.Hv, s.B);
    if (z != nullptr)
        prefill_chunk_kernel<true><<<grid, kThreads, kSmemBytes, st>>>(tk, tq, tv, tz, p);
    else
        prefill_chunk_kernel<false><<<grid, kThreads, kSmemBytes, st>>>(tk, tq, tv, tz, p);
    return cudaGetLastError();
}

}  // namespace gdn
