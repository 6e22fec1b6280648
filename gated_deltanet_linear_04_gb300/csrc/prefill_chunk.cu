// Chunked (WY / UT-transform) prefill on the 5th-generation tensor cores,
// single pass: one CTA (256 threads) owns one (b, hv) head for all T and
// walks its chunks of 64 steps in order, the f32 state resident in TMEM.  The
// products and their operand layouts are described in chunk_form.cuh; per
// chunk the phases are:
//   S1 base-2 log-decay prefix sums and step factors (warp 0)
//   S2 [K;Q] K^T on the tensor core while the tf32 operands gQ, Kc^T,
//      (b g K)^T, (b V)^T are built
//   S3 A from K K^T; the next chunk's q/k/v are prefetched by TMA
//   S4 T = (I + A)^-1 by blocked doubling (8x8 diagonal blocks, then 16-,
//      32-, 64-wide merges X = -T_bb A_ba T_aa) on the CUDA cores
//   S5 U^T, W^T; -W to shared memory
//   S6 S0 (-W)^T (into the W columns), Y^T = S0 (gQ)^T with S0 read from
//      TMEM; D^T = U^T + S0 (-W)^T is added in f32 in S7
//   S7 D^T and P = M o Q K^T to shared memory; S <- 2^lg_63 S
//   S8 Y^T += D^T P^T, S += D^T Kc^T
//   S9 y staged in shared memory as bf16 and stored by one TMA store of the
//      tile (3-D tensor map, clipped at the row's T)
// q, k, v tiles arrive by TMA (k and q 128B-swizzled straight into the
// MMA operand layout), prefetched one chunk ahead.  Head sizes Dk, Dv of 32,
// 64 or 128 all run on 128-wide tiles (chunk_form.cuh: the columns past the
// head read as zeros), so a chunk costs the same at every head size.
// Shared memory: 13 slots of 16 KiB reused across the phases of a chunk.
// Chunks whose 64 steps are all masked are skipped: their y is written zero and
// their inputs are never staged.
//
// NORM variant: each chunk's output is the layer's RMSNormGated of y ("mlex
// 0.1.2, src/models/gated_delta.rs", GatedDeltaNet::forward: f32 rms_norm of
// the bf16 y over Dv, times the norm weight, times silu(z), cast to bf16),
// computed from the bf16 y staging tile with the z tile brought in by TMA,
// so y itself never goes to memory.
#include "chunk_form.cuh"
#include "common.cuh"
#include "internal.h"
#include "mask_scan.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace chunkform;

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

constexpr uint32_t kTmemCols = 512;

struct ChunkParams {
    const float *g, *beta, *state_in;
    float *state_out;
    const uint8_t *mask;
    const int *order;   // row slot -> batch row (optional, with a mask)
    uint16_t *y;        // y, or the gated-norm output for the NORM variant
    const float *norm_w;
    float norm_eps;
    unsigned *err;
    int B, T, Hk, Hv, Dk, Dv;
    // optional records for the chunked backward (chunk_form.cuh layout, index
    // (b Hv + hv) nchunks + c): the state at every chunk's start, D^T of every chunk
    float *rec_s, *rec_d;
};

// REC: store the records of the chunked backward (p.rec_s, p.rec_d) instead
// of y, which the backward does not read
template <bool NORM, bool REC>
__global__ void __launch_bounds__(kThreads, 1) prefill_chunk_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                     const __grid_constant__ CUtensorMap tm_q,
                                                                     const __grid_constant__ CUtensorMap tm_v,
                                                                     const __grid_constant__ CUtensorMap tm_z,
                                                                     const __grid_constant__ CUtensorMap tm_y,
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
        for (int i = tid; i < kD; i += kThreads) s_w[i] = i < p.Dv ? p.norm_w[i] : 0.0f;
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
    state_to_tmem(p.state_in, tmem + lane_base + C_S, b, hv, p.Hv, p.Dk, p.Dv, row, half);

    // per-step g, beta, mask of a chunk: gathered into registers early (the
    // last two warps, one step per thread) and published to shared memory
    // later, so the global load latency never sits in front of a block
    // barrier; those warps also issue the next chunk's TMA, so that the first
    // two warps, which run A and the inverse's first phase, are not held up
    constexpr int kStepT0 = kThreads - kC;
    float pf_g = 1.0f, pf_b = 0.0f;
    int pf_m = 0;
    auto gather_steps = [&](int c) {
        pf_g = 1.0f;
        pf_b = 0.0f;
        pf_m = 0;
        const int i = tid - kStepT0;
        const int t = c * kC + i;
        if (i >= 0 && t < T) {
            const size_t gi = ((size_t)b * T + t) * p.Hv + hv;
            pf_m = p.mask == nullptr ? 1 : (p.mask[(size_t)b * T + t] != 0);
            if (pf_m) {
                pf_g = p.g[gi];
                pf_b = p.beta[gi];
            }
        }
    };
    auto publish_steps = [&](int slot) {
        const int i = tid - kStepT0;
        if (i >= 0) {
            s_g[slot][i] = pf_g;
            s_b[slot][i] = pf_b;
            s_m[slot][i] = pf_m;
        }
    };
    auto issue_tma = [&](int c) {
        if (tid == kThreads - 1)
            load_chunk_tiles(sm, S_KQ, S_V, &tm_k, &tm_q, &tm_v, p.Dk, p.Dv, hk, hv, b * T + c * kC, &bar_tma);
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
    uint16_t *y_row0 = p.y + (size_t)b * T * p.Hv * p.Dv + (size_t)hv * p.Dv;
    const size_t y_stride = (size_t)p.Hv * p.Dv;
    int c = scan.next_active(0);
    if constexpr (!REC) zero_y_rows(y_row0, y_stride, 0, min(c * kC, T), p.Dv);   // REC: y is not needed
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
        // ---- S1: chunk inputs, log-decay prefix sums (warp 0 for the first
        // chunk; later ones have them from the previous chunk's S8)
        ok = mbar_wait(&bar_tma, (uint32_t)(it & 1), p.err);
        if (it == 0 && warp == 0) step_factors(lane, s_g[st], s_b[st], s_lg, s_gam, s_kc, s_beta, s_bg);
        if (tid == 0) bulk_wait_read();   // the previous y store has read its tile (slot 9 is rebuilt below)
        ok = __syncthreads_and(ok) != 0;
        if (!ok) break;

        const int cn = scan.next_active(c + 1);
        if (cn < nchunks) gather_steps(cn);
        // ---- S2: [K;Q] K^T on the tensor core; meanwhile build the tf32 operands
        if (tid == 0) {
            umma::fence_after_sync();
            issue_kq(tmem, base, S_KQ);
            umma::mma_commit(&bar_mma);
        }
        build_gq(sm, S_KQ, S_GQ, s_gam, tid);
        build_kt_bk(sm, S_KQ, S_KT, S_BK, s_kc, s_bg, tid);
        build_bv(sm, S_V, S_BV, s_beta, tid);

        // ---- S3: A from K K^T (lanes 0-63)
        if (!wait_mma()) { ok = false; break; }
        if (quad < 2) build_a(tmem + lane_base + C_QK, As, s_lg, s_beta, row, half);
        // K and V tiles are no longer read: prefetch the next chunk
        umma::fence_before_sync();
        __syncthreads();
        if (cn < nchunks) {
            issue_tma(cn);
            publish_steps(st ^ 1);
        }

        // ---- S4: T = (I + A)^-1 by blocked doubling, in place in As
        invert_unit_lower(As, Ys, tid);
        t_to_tf32(As, sm, S_T, tid);   // the Y scratch is dead
        publish();

        // ---- S5: U^T and W^T on the tensor core
        if (tid == 0) {
            issue_uw(tmem, base, S_T, S_BV, S_BK);
            umma::mma_commit(&bar_mma);
        }
        if (!wait_mma()) { ok = false; break; }
        // -W -> smem (B operand of the D update)
        neg_w_tile(tmem + lane_base + C_W, sm, S_NW, row, half);
        publish();

        // ---- S6: S0 (-W)^T -> W columns ; Y^T = S0 (gQ)^T
        if (tid == 0) {
            // A = the f32 state itself, read from TMEM (used as tf32)
            issue_s0_products(tmem, base, S_NW, S_GQ);
            umma::mma_commit(&bar_mma);
        }
        if (!wait_mma()) { ok = false; break; }

        // ---- S7: D^T -> smem (A operand); P = M o Q K^T -> smem (B operand);
        // S <- 2^lg_63 S in TMEM (the D and Y products have read S already)
        if constexpr (NORM) {
            // the gQ slot is free now: bring in this chunk's z tile
            if (tid == 0) {
                mbar_expect_tx(&bar_z, 16384);
                load_chunk_z(sm + S_Z, &tm_z, p.Dv, hv, b * T + t0, &bar_z);
                z_pending = true;
                z_parity = (uint32_t)(it & 1);
            }
        }
        const size_t ci = ((size_t)b * p.Hv + hv) * nchunks + c;
        if constexpr (REC) decay_state(tmem + lane_base + C_S, s_gam[kC - 1], half, p.rec_s + ci * kRec128, row);
        else decay_state(tmem + lane_base + C_S, s_gam[kC - 1], half);
        {
            // the TMEM reads in flight before the one wait; D^T = U^T + S0 (-W)^T
            float dv[32], dp[32], qk[32];
            umma::tmem_ld32(tmem + lane_base + C_D + half * 32, dv);
            umma::tmem_ld32(tmem + lane_base + C_W + half * 32, dp);
            if (quad >= 2) umma::tmem_ld32(tmem + lane_base + C_QK + half * 32, qk);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) dv[j] += dp[j];
            dt_tile(dv, sm, S_DT, row, half);
            if (quad >= 2) p_tile(qk, sm, S_P, s_lg, row, half);
        }
        umma::tmem_st_wait();   // the decayed state is in TMEM before the product accumulates onto it
        publish();

        // ---- S8: Y^T += D^T P^T ; S += D^T Kc^T; while they run, warp 1
        // forms the next chunk's step factors (this chunk's are dead after S7)
        if (warp == 1 && cn < nchunks)
            step_factors(lane, s_g[st ^ 1], s_b[st ^ 1], s_lg, s_gam, s_kc, s_beta, s_bg);
        if (tid == 0) {
            issue_dt_products(tmem, base, S_DT, S_P, S_KT);
            umma::mma_commit(&bar_mma);
            if constexpr (REC) {
                // the D^T record: the operand tile itself, stored while the
                // products run (read out before the next chunk's S1 wait)
                bulk_store(p.rec_d + ci * kRec64, sm + S_DT, 32768);
                bulk_commit();
            }
        }
        if (!wait_mma()) { ok = false; break; }

        // ---- S9: y through a shared staging tile [64 steps][128 dv] bf16
        // (masked steps zero), then one TMA store of the tile clipped at T
        if constexpr (!REC) {
            stage_y(tmem + lane_base + C_Y, sm, S_YST, s_m[st], row, half);
            fence_proxy_async_smem();
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
            const float rs = 1.0f / sqrtf(ss * (1.0f / (float)p.Dv) + p.norm_eps);
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
            fence_proxy_async_smem();
            ok = __syncthreads_and(ok) != 0;
            if (!ok) break;
        }
        if constexpr (!REC) {
            if (tid == 0) {
                store_chunk_y(&tm_y, p.Dv, hv, t0, b, sm + S_YST);
                bulk_commit();
            }
            zero_y_rows(y_row0, y_stride, min((c + 1) * kC, T), min(cn * kC, T), p.Dv);
        }
        c = cn;
    }

    if (tid == 0) bulk_wait_read();   // the last y store has read its tile
    // ---- final state (only when every wait succeeded)
    if (__syncthreads_and(ok)) {
        state_from_tmem(p.state_out, tmem + lane_base + C_S, b, hv, p.Hv, p.Dk, p.Dv, row, half);
    } else if (tid == 0) {
        // a wait gave up: give in-flight MMAs (and a z copy) a bounded chance to drain
        mbar_wait(&bar_mma, mma_phase & 1u, nullptr);
        if (z_pending) mbar_wait(&bar_z, z_parity, nullptr);
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

template <bool NORM, bool REC>
cudaError_t set_smem_attr() {
    static unsigned long long attr_done = 0;   // per instantiation, one bit per device
    return set_max_smem(attr_done, prefill_chunk_kernel<NORM, REC>, kSmemBytes);
}

}  // namespace

cudaError_t launch_prefill_chunked(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                   const float *g, const float *beta, const float *state_in, float *state_out,
                                   const uint8_t *mask, const int *order, uint16_t *y, const uint16_t *z,
                                   const float *norm_w, float norm_eps, unsigned *err, cudaStream_t st,
                                   float *rec_s, float *rec_d) {
    if (s.Dk > kD || s.Dv > kD) return cudaErrorNotSupported;
    ChunkMaps m;
    if (!encode_chunk_maps(&m, s, q, k, v, z, y)) return cudaErrorInvalidValue;
    const bool rec = rec_s != nullptr && rec_d != nullptr;
    if (rec && z != nullptr) return cudaErrorNotSupported;
    cudaError_t e = z != nullptr ? set_smem_attr<true, false>()
                                 : (rec ? set_smem_attr<false, true>() : set_smem_attr<false, false>());
    if (e != cudaSuccess) return e;
    ChunkParams p{g, beta, state_in, state_out, mask, mask != nullptr ? order : nullptr, y, norm_w, norm_eps, err,
                  s.B, s.T, s.Hk, s.Hv, s.Dk, s.Dv, rec_s, rec_d};
    dim3 grid(s.Hv, s.B);
    if (z != nullptr)
        prefill_chunk_kernel<true, false><<<grid, kThreads, kSmemBytes, st>>>(m.k, m.q, m.v, m.z, m.y, p);
    else if (rec)
        prefill_chunk_kernel<false, true><<<grid, kThreads, kSmemBytes, st>>>(m.k, m.q, m.v, m.z, m.y, p);
    else
        prefill_chunk_kernel<false, false><<<grid, kThreads, kSmemBytes, st>>>(m.k, m.q, m.v, m.z, m.y, p);
    return cudaGetLastError();
}

}  // namespace gdn
