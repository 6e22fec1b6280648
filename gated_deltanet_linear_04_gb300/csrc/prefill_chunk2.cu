// Chunked (WY / UT-transform) prefill in two passes, for batches with fewer
// heads than the GPU has SMs.
//
// In the single-pass kernel one CTA walks all chunks of its head in order, so
// with few heads (one sequence of 32 heads on 152 SMs) most SMs idle and the
// serial chain of chunks sets the time.  Most of a chunk's work does not
// depend on the state: the step factors, the operand builds, A, the inverse
// T = (I + A)^-1, U^T, W^T and P (the products of chunk_form.cuh that do not
// read S0).  Pass 1 ("prep") does that work for every (b, hv, chunk) and
// writes the results to the workspace as images of the shared-memory tiles
// the products read.  Pass 2 ("state") keeps one CTA per head walking the
// chunks in order, but per chunk it only bulk-copies the images back and runs
// the state products (S0 (-W)^T and Y^T = S0 (gQ)^T, D^T = U^T + S0 (-W)^T
// added in f32, then Y^T += D^T P^T and S += D^T Kc^T) and the output.
// Both passes run the single-pass kernel's arithmetic on the same operand
// bits, so y and the state are bit-identical to it.
//
// Two launch forms:
//   * separate: the prep kernel (one CTA per chunk, whole GPU), then the state
//     kernel (one CTA per head);
//   * overlapped, when the heads take at most a quarter of the SMs: one
//     cooperative launch of one CTA per SM (all resident at once) in which the
//     first B*Hv CTAs run the state chains while the others produce the chunk
//     images in chunk order; each image is published with a ready flag
//     (bulk stores complete, proxy fence, release store) that the state CTA
//     acquires before its bulk load.  A producer fetches its next unit's
//     tiles while the current unit finishes, and publishes a unit once the
//     next one has done its operand builds, so it never waits for its own
//     stores to land.  Every wait is bounded and sets the device error word
//     if it gives up.
//
// Workspace blob per (b, hv, chunk), laid out like pass 2's shared memory so
// that one 1-D bulk copy brings in each group:
//   group A  [-W | gQ 64 KiB][U^T 32 KiB][meta 1 KiB: 2^lg_63]
//   group B  [P | Kc^T 48 KiB]
// -W and gQ are interleaved by K-tile (-W's 64 rows, then gQ's 64 rows, of
// each 32-column tile) so that together they are one N = 128 B operand, and
// P and Kc^T likewise (P's 64 rows, then Kc^T's 128) one N = 192 operand:
// pass 2 runs the two products that read S0 as one MMA per K step into the
// adjacent D and Y accumulators, and the two that read D^T as one into the
// adjacent Y and S accumulators.
// U^T is plain f32 [128 dv][64 steps] with each row's 16-byte groups permuted
// (group j stored at j ^ (dv % 16)) so that a warp's row-per-thread accesses
// spread over the banks.  After the blobs come the ready flags (one int per
// blob).  Wholly masked chunks are skipped by both passes.
#include "chunk_form.cuh"
#include "common.cuh"
#include "internal.h"
#include "mask_scan.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace chunkform;

// blob layout
constexpr uint32_t B_NWGQ = 0, B_UT = 65536, B_META = 98304;   // [-W_kt 8 KiB | gQ_kt 8 KiB] x 4
constexpr uint32_t kGroupA = 98304 + 1024;
constexpr uint32_t B_PKT = kGroupA;                            // [P_kt 8 KiB | Kc^T_kt 16 KiB] x 2
constexpr uint32_t kGroupB = 32768 + 16384;
constexpr size_t kBlobBytes = (size_t)kGroupA + kGroupB;

// pass 1 shared memory: 13 slots of 16 KiB in one of two maps.  A unit's k/q
// and v tiles arrive in its KQ (two slots) and V slots; once the products
// have read them, KQ and V hold P and U^T and (bV)^T holds -W.  Each output
// leaves by bulk stores once it is final (gQ and Kc^T after the builds, P
// after its tile, -W and U^T at the unit's end), so that the next unit, whose
// builds overwrite these slots, waits only for the last 64 KiB to be read
// out.  The BK pair and the A slot are free at the end of a unit, and the
// next unit's k/q and v tiles are fetched into them as soon as the U/W
// products complete, so the two maps alternate:
//   map 0: KQ 6-7, V 8,  gQ 0-1, Kc^T 2-3, bV 4-5, bK 9-10, A 11, T 12
//   map 1: KQ 9-10, V 11, gQ 0-1, Kc^T 2-3, bV 4-5, bK 6-7,  A 8,  T 12
// (map 0's bK/A are map 1's KQ/V and the other way round).  Every other
// slot of a unit is one of the previous unit's outputs or T, written only
// after the previous stores have read them out.
struct PrepMap {
    uint32_t kq, v, gq, kt, bv, bk, a, t;
};
__device__ __forceinline__ PrepMap prep_map(int parity) {
    return parity == 0 ? PrepMap{6 * kSlot, 8 * kSlot, 0, 2 * kSlot, 4 * kSlot, 9 * kSlot, 11 * kSlot, 12 * kSlot}
                       : PrepMap{9 * kSlot, 11 * kSlot, 0, 2 * kSlot, 4 * kSlot, 6 * kSlot, 8 * kSlot, 12 * kSlot};
}
constexpr uint32_t kP1Smem = 13 * kSlot + 1024;

// pass 2 shared memory: group A and group B images, then D^T and y staging
constexpr uint32_t P2_NWGQ = B_NWGQ, P2_UT = B_UT, P2_META = B_META;
constexpr uint32_t P2_PKT = B_PKT;
constexpr uint32_t P2_DT = kGroupA + kGroupB;            // 32 KiB
constexpr uint32_t P2_YST = P2_DT + 32768;               // 16 KiB
constexpr uint32_t kP2Smem = P2_YST + 16384 + 1024;
constexpr uint32_t kFusedSmem = kP1Smem > kP2Smem ? kP1Smem : kP2Smem;

struct TwoPassParams {
    const float *g, *beta, *state_in;
    float *state_out;
    const uint8_t *mask;
    const int *order;   // row slot -> batch row (optional, with a mask)
    uint16_t *y;
    uint8_t *blobs;
    int *ready;         // overlapped form: one flag per blob (zeroed before launch); else null
    unsigned *err;
    int B, T, Hk, Hv, Dk, Dv, nchunks;
    // optional records for the chunked backward (chunk_form.cuh layout, one
    // per blob index): the state at every chunk's start and D^T of every chunk
    float *rec_s, *rec_d;
};

// Static shared memory of both roles.
struct TwoPassShared {
    uint64_t bar0, bar1, bar2;   // prep: TMA, MMA.  state: group A, group B, MMA
    uint32_t tmem_slot;
    float s_g[kC], s_b[kC];
    __align__(16) float s_lg[kC];
    __align__(16) float s_gam[kC];
    __align__(16) float s_beta[kC];
    __align__(16) float s_bg[kC];
    __align__(16) float s_kc[kC];
    int s_m[2][kC];
    uint32_t scan_bits[ChunkScan<kThreads>::kWords];
};

__device__ __forceinline__ size_t blob_index(const TwoPassParams &p, int b, int hv, int c) {
    return ((size_t)b * p.Hv + hv) * p.nchunks + c;
}

// U^T row of thread `row`, 16-byte group j, in the permuted plain layout
__device__ __forceinline__ uint32_t ut_off(int row, int j) { return (uint32_t)(row * 256 + ((j ^ (row & 15)) * 16)); }

// Publish a blob whose bulk stores this thread has seen complete: order the
// async-proxy writes before a release store of the flag.
__device__ __forceinline__ void publish_ready(int *flag) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}

// Bounded wait (acquire) for a blob's flag, then order it before the
// async-proxy bulk load that reads the blob.
__device__ __forceinline__ bool wait_ready(const int *flag, unsigned *err) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v != 0) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            return true;
        }
        __nanosleep(64);
    }
    if (err) atomicOr(err, kErrMbarTimeout);
    return false;
}

// ---------------------------------------------------------------------------
// pass 1: the state-independent part of chunk c of head (b, hv), one unit of a
// producer's sequence.  The producer keeps across its units: the TMA and MMA
// barrier phases, the gates of the current unit (threads < 64, in registers),
// whether the previous unit's stores are still to be published, and which
// map the current unit uses.
// ---------------------------------------------------------------------------
struct Producer {
    uint32_t tma_phase = 0, mma_phase = 0;
    int parity = 0;
    float gg = 1.0f, bb = 0.0f;   // this thread's step of the current unit (threads < 64)
    int *pending_flag = nullptr;  // ready flag of the previous unit, published once its stores are complete
    bool tma_pending = false;     // thread 0: a prefetch is in flight
};

// Gates (and whether the chunk holds a valid step) of unit (c, b, hv) into
// this thread's registers; returns whether the chunk holds a valid step
// (block-wide when there is a mask).
__device__ __forceinline__ bool unit_gates(const TwoPassParams &p, int c, int b, int hv, float &gg, float &bb) {
    const int tid = threadIdx.x, t = c * kC + tid;
    gg = 1.0f;
    bb = 0.0f;
    int m = 0;
    if (tid < kC && t < p.T) {
        const size_t gi = ((size_t)b * p.T + t) * p.Hv + hv;
        m = p.mask == nullptr ? 1 : (p.mask[(size_t)b * p.T + t] != 0);
        if (m) {
            gg = p.g[gi];
            bb = p.beta[gi];
        }
    }
    return p.mask == nullptr ? true : __syncthreads_or(m) != 0;
}

// k/q and v tiles of unit (c, b, hv) into the KQ and V slots of `m` (thread 0)
__device__ __forceinline__ void unit_tiles(const TwoPassParams &p, const CUtensorMap *tm_k, const CUtensorMap *tm_q,
                                           const CUtensorMap *tm_v, TwoPassShared &sh, uint8_t *sm,
                                           const PrepMap &m, int c, int b, int hv) {
    load_chunk_tiles(sm, m.kq, m.v, tm_k, tm_q, tm_v, p.Dk, p.Dv, hv / (p.Hv / p.Hk), hv, b * p.T + c * kC, &sh.bar0);
}

// Publishes the previous unit's image once its stores have completed (thread
// 0).  Inside a unit the newest store group is that unit's own gQ / Kc^T,
// which need not be waited for.
__device__ __forceinline__ void publish_pending(Producer &pr, bool own_group_pending) {
    if (pr.pending_flag != nullptr) {
        // the writes are done, not only read out
        if (own_group_pending) bulk_wait_all_but_newest();
        else bulk_wait_all();
        __threadfence();    // ... and so is the meta store
        publish_ready(pr.pending_flag);
        pr.pending_flag = nullptr;
    }
}

// One unit.  Its k/q/v tiles are in flight on sh.bar0 into the KQ/V slots of
// map pr.parity and its gates are in pr.gg/pr.bb.  `next` (c, b, hv; c < 0
// for none) is the producer's next unit: its tiles are fetched once this
// unit's U/W products have completed.  Returns false if a wait gave up.
// Ends with a block barrier; the unit's stores are committed, and with ready
// flags their publication is left to the next unit (or publish_pending).
__device__ __forceinline__ bool prep_unit(const TwoPassParams &p, const CUtensorMap *tm_k, const CUtensorMap *tm_q,
                                          const CUtensorMap *tm_v, TwoPassShared &sh, uint8_t *sm, uint32_t base,
                                          uint32_t tmem, Producer &pr, int c, int b, int hv, int nc, int nb,
                                          int nhv) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2, row = quad * 32 + lane;
    const uint32_t lane_tmem = tmem + ((uint32_t)(quad * 32) << 16);
    const PrepMap M = prep_map(pr.parity);
    float *As = reinterpret_cast<float *>(sm + M.a);
    float *Ys = reinterpret_cast<float *>(sm + M.t);

    if (tid < kC) {
        sh.s_g[tid] = pr.gg;
        sh.s_b[tid] = pr.bb;
    }
    // the previous unit's outputs (this unit's gQ ... T slots) have been read out
    if (tid == 0) bulk_wait_read();

    auto wait_mma = [&]() {
        bool w = mbar_wait(&sh.bar1, pr.mma_phase & 1u, p.err);
        ++pr.mma_phase;
        w = __syncthreads_and(w) != 0;
        umma::fence_after_sync();
        return w;
    };
    auto publish = [&]() {
        fence_proxy_async_smem();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
    };

    bool ok = mbar_wait(&sh.bar0, pr.tma_phase & 1u, p.err);
    ++pr.tma_phase;
    if (tid == 0) pr.tma_pending = false;
    __syncthreads();   // gates in shared memory, the previous stores read out
    if (warp == 0) step_factors(lane, sh.s_g, sh.s_b, sh.s_lg, sh.s_gam, sh.s_kc, sh.s_beta, sh.s_bg);
    ok = __syncthreads_and(ok) != 0;
    if (ok) {
        if (tid == 0) {
            umma::fence_after_sync();
            issue_kq(tmem, base, M.kq);
            umma::mma_commit(&sh.bar1);
        }
        build_gq(sm, M.kq, M.gq, sh.s_gam, tid);
        build_kt_bk(sm, M.kq, M.kt, M.bk, sh.s_kc, sh.s_bg, tid);
        build_bv(sm, M.v, M.bv, sh.s_beta, tid);
        fence_proxy_async_smem();   // gQ and Kc^T leave now (below), not with the rest
        ok = wait_mma();
    }
    uint8_t *const blob = p.blobs + blob_index(p, b, hv, c) * kBlobBytes;
    if (ok && tid == 0) {
        // gQ and Kc^T are final: store them while the unit goes on, so that
        // only -W and U^T are left for the unit's end
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) bulk_store(blob + B_NWGQ + kt * 16384 + 8192, sm + M.gq + kt * 8192, 8192);
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) bulk_store(blob + B_PKT + kt * 24576 + 8192, sm + M.kt + kt * kSlot, 16384);
        bulk_commit();
    }
    if (ok) {
        // A from K K^T (quads 0-1); P from Q K^T (quads 2-3) into the dead KQ slot
        if (quad < 2) {
            build_a(lane_tmem + C_QK, As, sh.s_lg, sh.s_beta, row, half);
        } else {
            float qk[32];
            umma::tmem_ld32(lane_tmem + C_QK + half * 32, qk);
            umma::tmem_ld_wait();
            p_tile(qk, sm, M.kq, sh.s_lg, row, half);
        }
        fence_proxy_async_smem();   // P leaves as soon as it is written
        // the previous unit's stores have had this unit's builds to complete
        if (tid == 0) publish_pending(pr, true);
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int kt = 0; kt < 2; ++kt) bulk_store(blob + B_PKT + kt * 24576, sm + M.kq + kt * 8192, 8192);
            bulk_commit();
        }
        invert_unit_lower(As, Ys, tid);
        t_to_tf32(As, sm, M.t, tid);
        publish();
        if (tid == 0) {
            issue_uw(tmem, base, M.t, M.bv, M.bk);
            umma::mma_commit(&sh.bar1);
        }
        ok = wait_mma();
    }
    if (ok) {
        // bK and A are free: fetch the next unit's tiles there (the next map's KQ and V)
        if (tid == 0 && nc >= 0) {
            unit_tiles(p, tm_k, tm_q, tm_v, sh, sm, prep_map(pr.parity ^ 1), nc, nb, nhv);
            pr.tma_pending = true;
        }
        neg_w_tile(lane_tmem + C_W, sm, M.bv, row, half);
        float uv[32];
        umma::tmem_ld32(lane_tmem + C_D + half * 32, uv);
        umma::tmem_ld_wait();
        const uint32_t ut = M.kq + kSlot;   // U^T: the KQ pair's second slot and the V slot
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
            *reinterpret_cast<float4 *>(sm + ut + ut_off(row, half * 8 + jj)) =
                make_float4(uv[4 * jj], uv[4 * jj + 1], uv[4 * jj + 2], uv[4 * jj + 3]);
        fence_proxy_async_smem();
        umma::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            *reinterpret_cast<float *>(blob + B_META) = sh.s_gam[kC - 1];
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) bulk_store(blob + B_NWGQ + kt * 16384, sm + M.bv + kt * 8192, 8192);
            bulk_store(blob + B_UT, sm + ut, 32768);
            bulk_commit();
            if (p.ready != nullptr) pr.pending_flag = p.ready + blob_index(p, b, hv, c);
        }
    } else if (tid == 0) {
        // a wait gave up: give in-flight MMAs and copies a bounded chance to drain
        mbar_wait(&sh.bar1, pr.mma_phase & 1u, nullptr);
        if (pr.tma_pending) mbar_wait(&sh.bar0, pr.tma_phase & 1u, nullptr);
    }
    pr.parity ^= 1;
    umma::fence_before_sync();
    __syncthreads();
    return ok;
}

// ---------------------------------------------------------------------------
// pass 2 TMEM columns: D | Y | S adjacent, so that
//   [D'^T | Y^T] = S0 [-W ; gQ]^T                    (N = 128, K = 128)
//   [Y^T | S]  += D^T [P ; Kc^T]^T                    (N = 192, K = 64)
// run as one MMA per K step each, S0 read from TMEM (tf32 by truncation),
// with D^T = U^T + D'^T added in f32 as the D^T tile is built.  Each
// accumulator sees its MMAs in the single pass's order and the addition is
// the single pass's, so the results match it bit for bit.
// ---------------------------------------------------------------------------
constexpr uint32_t C2_D = 64, C2_Y = 128, C2_S = 192;

__device__ __forceinline__ void issue_s0_merged(uint32_t tmem, uint32_t base) {
    const uint32_t id = umma::idesc(128, 128, umma::kFmtTF32);
#pragma unroll
    for (int k = 0; k < 16; ++k)
        umma::mma_tf32_tmem_a(tmem + C2_D, tmem + C2_S + 8 * k,
                              umma::desc_sw128(base + P2_NWGQ + (k >> 2) * 16384 + (k & 3) * 32), id, k > 0);
}

__device__ __forceinline__ void issue_dt_merged(uint32_t tmem, uint32_t base) {
    const uint32_t id = umma::idesc(128, 192, umma::kFmtTF32);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t kt = k >> 2, ko = (k & 3) * 32;
        umma::mma_tf32(tmem + C2_Y, umma::desc_sw128(base + P2_DT + kt * kSlot + ko),
                       umma::desc_sw128(base + P2_PKT + kt * 24576 + ko), id, true);
    }
}

// ---------------------------------------------------------------------------
// pass 2: the chunk chain of head (b, hv), state products only.  The caller
// has initialised sh.bar0-2 and allocated 512 TMEM columns.
// ---------------------------------------------------------------------------
// REC: store the records of the chunked backward (p.rec_s, p.rec_d) instead
// of y, which the backward does not read
template <bool REC>
__device__ __forceinline__ void state_head(const TwoPassParams &p, const CUtensorMap *tm_y, TwoPassShared &sh,
                                           uint8_t *sm, uint32_t base, uint32_t tmem, int b, int hv) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2, row = quad * 32 + lane;
    const int T = p.T;
    const int nchunks = p.nchunks;
    const uint32_t lane_tmem = tmem + ((uint32_t)(quad * 32) << 16);

    // initial state -> TMEM S (row = dv, columns = dk); half 0: dk 0-63, half 1: 64-127
    state_to_tmem(p.state_in, lane_tmem + C2_S, b, hv, p.Hv, p.Dk, p.Dv, row, half);
    (void)lane;

    int pf_m = 0;
    auto gather_mask = [&](int c) {
        const int t = c * kC + tid;
        pf_m = (tid < kC && t < T) ? (p.mask == nullptr ? 1 : (p.mask[(size_t)b * T + t] != 0)) : 0;
    };
    // thread 0 only: outstanding copies, for the drain after a failed wait;
    // after one flag wait has given up (error word set) no further one is made,
    // so a failed producer costs one bounded wait, not one per chunk
    bool a_pending = false, b_pending = false, flag_gave_up = false;
    uint32_t a_parity = 0, b_parity = 0;
    auto load_a = [&](int c, int it) {
        if (tid == 0) {
            const size_t bi = blob_index(p, b, hv, c);
            if (p.ready != nullptr && !flag_gave_up) flag_gave_up = !wait_ready(p.ready + bi, p.err);
            mbar_expect_tx(&sh.bar0, kGroupA);
            bulk_load(sm + P2_NWGQ, p.blobs + bi * kBlobBytes, kGroupA, &sh.bar0);
            a_pending = true;
            a_parity = (uint32_t)(it & 1);
        }
    };
    auto load_b = [&](int c, int it) {
        if (tid == 0) {
            // group B of chunk c is loaded after group A, whose flag covers the whole blob
            mbar_expect_tx(&sh.bar1, kGroupB);
            bulk_load(sm + P2_PKT, p.blobs + blob_index(p, b, hv, c) * kBlobBytes + kGroupA, kGroupB, &sh.bar1);
            b_pending = true;
            b_parity = (uint32_t)(it & 1);
        }
    };

    uint32_t mma_phase = 0;
    bool ok = true;
    auto wait_mma = [&]() {
        bool w = mbar_wait(&sh.bar2, mma_phase & 1u, p.err);
        ++mma_phase;
        w = __syncthreads_and(w) != 0;
        umma::fence_after_sync();
        return w;
    };
    auto publish = [&]() {
        fence_proxy_async_smem();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
    };

    ChunkScan<kThreads> scan(p.mask == nullptr ? nullptr : p.mask + (size_t)b * T, T, sh.scan_bits);
    uint16_t *y_row0 = p.y + (size_t)b * T * p.Hv * p.Dv + (size_t)hv * p.Dv;
    const size_t y_stride = (size_t)p.Hv * p.Dv;
    int c = scan.next_active(0);
    if constexpr (!REC) zero_y_rows(y_row0, y_stride, 0, min(c * kC, T), p.Dv);   // REC: y is not needed
    if (c < nchunks) {
        load_a(c, 0);
        load_b(c, 0);
        gather_mask(c);
        if (tid < kC) sh.s_m[0][tid] = pf_m;
    }
    umma::fence_before_sync();   // the initial state's TMEM stores, before the first product
    __syncthreads();

    for (int it = 0; c < nchunks && ok; ++it) {
        const int st = it & 1;
        const int t0 = c * kC;
        // every thread waits for group A itself; the block agrees on the
        // outcome at the product's wait below (no barrier of its own here)
        const bool got_a = mbar_wait(&sh.bar0, (uint32_t)(it & 1), p.err);
        if (tid == 0) a_pending = false;
        const int cn = scan.next_active(c + 1);
        if (cn < nchunks) gather_mask(cn);

        // [D'^T | Y^T] = S0 [-W ; gQ]^T (the previous chunk's TMEM reads were
        // ordered before the barrier that ended it); while it runs, this
        // thread's U^T row comes out of the image, which the next chunk's
        // group A overwrites
        const float gl = *reinterpret_cast<const float *>(sm + P2_META);
        if (tid == 0 && got_a) {
            umma::fence_after_sync();
            issue_s0_merged(tmem, base);
            umma::mma_commit(&sh.bar2);
            if constexpr (REC) bulk_wait_read();   // the previous D^T record has read the tile rewritten below
        }
        float ut[32];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const float4 v = *reinterpret_cast<const float4 *>(sm + P2_UT + ut_off(row, half * 8 + jj));
            ut[4 * jj] = v.x; ut[4 * jj + 1] = v.y; ut[4 * jj + 2] = v.z; ut[4 * jj + 3] = v.w;
        }
        {
            // thread 0 issued nothing if its wait gave up: then nobody waits
            // on the product's barrier
            const bool all_a = __syncthreads_and(got_a) != 0;
            if (!all_a) {
                if (tid == 0 && got_a) mbar_wait(&sh.bar2, mma_phase & 1u, nullptr);   // drain what was issued
                ok = false;
                break;
            }
        }
        if (!wait_mma()) { ok = false; break; }
        // group A has been consumed: fetch the next chunk's
        if (cn < nchunks) load_a(cn, it + 1);

        const size_t ci = blob_index(p, b, hv, c);
        if constexpr (REC) decay_state(lane_tmem + C2_S, gl, half, p.rec_s + ci * kRec128, row);
        else decay_state(lane_tmem + C2_S, gl, half);
        {
            float dv[32];
            umma::tmem_ld32(lane_tmem + C2_D + half * 32, dv);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) dv[j] = ut[j] + dv[j];   // D^T = U^T + S0 (-W)^T, as the single pass adds
            dt_tile(dv, sm, P2_DT, row, half);
        }
        umma::tmem_st_wait();   // the decayed state is in TMEM before the product accumulates onto it
        // group B waited for by every thread, and the D^T tile published,
        // at one barrier
        {
            const bool got_b = mbar_wait(&sh.bar1, (uint32_t)(it & 1), p.err);
            fence_proxy_async_smem();
            umma::fence_before_sync();
            ok = __syncthreads_and(got_b) != 0;
            umma::fence_after_sync();
        }
        if (tid == 0) b_pending = false;
        if (!ok) break;
        if (tid == 0) {
            umma::fence_after_sync();
            issue_dt_merged(tmem, base);
            umma::mma_commit(&sh.bar2);
            if constexpr (REC) {
                // the D^T record: the operand tile itself, stored while the
                // product runs (read out before the next chunk rewrites it)
                bulk_store(p.rec_d + ci * kRec64, sm + P2_DT, 32768);
                bulk_commit();
            } else {
                bulk_wait_read();   // the previous chunk's y store has read the staging tile
            }
        }
        if (!wait_mma()) { ok = false; break; }
        if (cn < nchunks) load_b(cn, it + 1);

        // y: the staged tile leaves by one TMA store (clipped at T), which
        // the next chunk's staging waits for
        if constexpr (!REC) {
            stage_y(lane_tmem + C2_Y, sm, P2_YST, sh.s_m[st], row, half);
            fence_proxy_async_smem();
        }
        umma::fence_before_sync();
        __syncthreads();
        if constexpr (!REC) {
            if (tid == 0) {
                store_chunk_y(tm_y, p.Dv, hv, t0, b, sm + P2_YST);
                bulk_commit();
            }
        }
        if (tid < kC) sh.s_m[st ^ 1][tid] = pf_m;
        if constexpr (!REC) zero_y_rows(y_row0, y_stride, min((c + 1) * kC, T), min(cn * kC, T), p.Dv);
        c = cn;
    }

    if (tid == 0) bulk_wait_read();   // the last y store has read the staging tile
    if (__syncthreads_and(ok)) {
        state_from_tmem(p.state_out, lane_tmem + C2_S, b, hv, p.Hv, p.Dk, p.Dv, row, half);
    } else if (tid == 0) {
        // a wait gave up: give in-flight MMAs and copies a bounded chance to drain
        mbar_wait(&sh.bar2, mma_phase & 1u, nullptr);
        if (a_pending) mbar_wait(&sh.bar0, a_parity, nullptr);
        if (b_pending) mbar_wait(&sh.bar1, b_parity, nullptr);
    }
    umma::fence_before_sync();
    __syncthreads();
}

// ---------------------------------------------------------------------------
// kernels
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint8_t *aligned_base(uint8_t *raw, uint32_t &base) {
    base = (smem_u32(raw) + 1023u) & ~1023u;
    return raw + (base - smem_u32(raw));
}

// barriers and TMEM of a CTA; returns the TMEM base
__device__ __forceinline__ uint32_t cta_setup(TwoPassShared &sh, uint32_t tmem_cols) {
    if (threadIdx.x == 0) {
        mbar_init(&sh.bar0, 1);
        mbar_init(&sh.bar1, 1);
        mbar_init(&sh.bar2, 1);
        fence_mbar_init();
    }
    if ((threadIdx.x >> 5) == 0) {
        umma::tmem_alloc(&sh.tmem_slot, tmem_cols);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    return sh.tmem_slot;
}

__device__ __forceinline__ void cta_teardown(uint32_t tmem, uint32_t tmem_cols) {
    if ((threadIdx.x >> 5) == 0) umma::tmem_dealloc(tmem, tmem_cols);
}

// separate form, pass 1: one CTA per (chunk, hv, b)
__global__ void __launch_bounds__(kThreads, 1) chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                  const __grid_constant__ CUtensorMap tm_q,
                                                                  const __grid_constant__ CUtensorMap tm_v,
                                                                  const TwoPassParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ TwoPassShared sh;
    uint32_t base;
    uint8_t *sm = aligned_base(smem_raw, base);
    const uint32_t tmem = cta_setup(sh, 256);
    Producer pr;
    const int c = blockIdx.x, b = blockIdx.z, hv = blockIdx.y;
    if (unit_gates(p, c, b, hv, pr.gg, pr.bb)) {
        if (threadIdx.x == 0) unit_tiles(p, &tm_k, &tm_q, &tm_v, sh, sm, prep_map(0), c, b, hv);
        prep_unit(p, &tm_k, &tm_q, &tm_v, sh, sm, base, tmem, pr, c, b, hv, -1, 0, 0);
        if (threadIdx.x == 0) bulk_wait_read();   // the stores have read shared memory
    }
    cta_teardown(tmem, 256);
}

// separate form, pass 2: one CTA per (hv, row slot)
template <bool REC>
__global__ void __launch_bounds__(kThreads, 1) chunk_state_kernel(const __grid_constant__ CUtensorMap tm_y,
                                                                   const TwoPassParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ TwoPassShared sh;
    uint32_t base;
    uint8_t *sm = aligned_base(smem_raw, base);
    const uint32_t tmem = cta_setup(sh, 512);
    const int b = p.order != nullptr ? p.order[blockIdx.y] : (int)blockIdx.y;
    state_head<REC>(p, &tm_y, sh, sm, base, tmem, b, blockIdx.x);
    cta_teardown(tmem, 512);
}

// overlapped form (cooperative launch, all CTAs resident): CTAs [0, n_heads)
// run the state chains, the others produce the chunk images in chunk order
template <bool REC>
__global__ void __launch_bounds__(kThreads, 1) chunk_overlap_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                     const __grid_constant__ CUtensorMap tm_q,
                                                                     const __grid_constant__ CUtensorMap tm_v,
                                                                     const __grid_constant__ CUtensorMap tm_y,
                                                                     const TwoPassParams p, const int n_heads) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ TwoPassShared sh;
    uint32_t base;
    uint8_t *sm = aligned_base(smem_raw, base);
    const bool is_state = (int)blockIdx.x < n_heads;
    const uint32_t cols = is_state ? 512u : 256u;
    const uint32_t tmem = cta_setup(sh, cols);
    if (is_state) {
        const int slot = blockIdx.x / p.Hv, hv = blockIdx.x % p.Hv;
        const int b = p.order != nullptr ? p.order[slot] : slot;
        state_head<REC>(p, &tm_y, sh, sm, base, tmem, b, hv);
    } else {
        // producer: units u = (chunk u / n_heads, head u % n_heads) in steps of
        // the producer count; wholly masked chunks are passed over
        const int n_prep = (int)gridDim.x - n_heads;
        const long n_units = (long)p.nchunks * n_heads;
        Producer pr;
        float ng = 1.0f, nb = 0.0f;
        // the first unit of `from` or after it that holds a valid step, its gates in (ng, nb)
        auto next_active = [&](long from) {
            long v = from;
            for (; v < n_units; v += n_prep) {
                const int h = (int)(v % n_heads);
                if (unit_gates(p, (int)(v / n_heads), h / p.Hv, h % p.Hv, ng, nb)) break;
            }
            return v;
        };
        long u = next_active((long)blockIdx.x - n_heads);
        if (u < n_units && threadIdx.x == 0) {
            const int h = (int)(u % n_heads);
            unit_tiles(p, &tm_k, &tm_q, &tm_v, sh, sm, prep_map(0), (int)(u / n_heads), h / p.Hv, h % p.Hv);
        }
        while (u < n_units) {
            pr.gg = ng;
            pr.bb = nb;
            const long un = next_active(u + n_prep);
            const int h = (int)(u % n_heads), hn = (int)(un % n_heads);
            const bool more = un < n_units;
            if (!prep_unit(p, &tm_k, &tm_q, &tm_v, sh, sm, base, tmem, pr, (int)(u / n_heads), h / p.Hv, h % p.Hv,
                           more ? (int)(un / n_heads) : -1, more ? hn / p.Hv : 0, more ? hn % p.Hv : 0))
                break;
            u = un;
        }
        if (threadIdx.x == 0) {
            publish_pending(pr, false);   // the last unit's image
            bulk_wait_read();
        }
    }
    cta_teardown(tmem, cols);
}

size_t blob_count(const Sizes &s) { return (size_t)s.B * s.Hv * (((size_t)s.T + kC - 1) / kC); }

}  // namespace

size_t prefill_two_pass_workspace(const Sizes &s) {
    const size_t n = blob_count(s);
    return n * kBlobBytes + ((n * sizeof(int) + 255) & ~(size_t)255);
}

bool prefill_two_pass_pays(const Sizes &s) { return (long)s.B * s.Hv < num_sms(); }

cudaError_t launch_prefill_two_pass(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                    const float *g, const float *beta, const float *state_in, float *state_out,
                                    const uint8_t *mask, const int *order, uint16_t *y, void *blobs,
                                    unsigned *err, cudaStream_t st, float *rec_s, float *rec_d) {
    if (s.Dk > kD || s.Dv > kD) return cudaErrorNotSupported;
    ChunkMaps m;
    if (!encode_chunk_maps(&m, s, q, k, v, nullptr, y)) return cudaErrorInvalidValue;
    const CUtensorMap &tk = m.k, &tq = m.q, &tv = m.v, &ty = m.y;
    const bool rec = rec_s != nullptr && rec_d != nullptr;
    static unsigned long long set1 = 0, set2 = 0, set3 = 0, set4 = 0, set5 = 0;   // one bit per device
    cudaError_t e = set_max_smem(set1, chunk_prep_kernel, kP1Smem);
    if (e == cudaSuccess)
        e = rec ? set_max_smem(set4, chunk_state_kernel<true>, kP2Smem)
                : set_max_smem(set2, chunk_state_kernel<false>, kP2Smem);
    if (e == cudaSuccess)
        e = rec ? set_max_smem(set5, chunk_overlap_kernel<true>, kFusedSmem)
                : set_max_smem(set3, chunk_overlap_kernel<false>, kFusedSmem);
    if (e != cudaSuccess) return e;
    const int nchunks = (s.T + kC - 1) / kC;
    const int n_heads = s.B * s.Hv;
    const size_t n_blobs = blob_count(s);
    TwoPassParams p{g, beta, state_in, state_out, mask, mask != nullptr ? order : nullptr, y,
                    static_cast<uint8_t *>(blobs), nullptr, err, s.B, s.T, s.Hk, s.Hv, s.Dk, s.Dv, nchunks,
                    rec_s, rec_d};

    // Overlapped form when the producers (all SMs but the heads') outnumber
    // the heads about three to one: a chunk image takes the producers roughly
    // three times as long as the state pass takes to consume one.
    int per_sm = 0;
    if (4 * n_heads <= num_sms() &&
        (rec ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chunk_overlap_kernel<true>, kThreads,
                                                             kFusedSmem)
             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chunk_overlap_kernel<false>, kThreads,
                                                             kFusedSmem)) == cudaSuccess &&
        per_sm >= 1) {
        p.ready = reinterpret_cast<int *>(static_cast<uint8_t *>(blobs) + n_blobs * kBlobBytes);
        e = cudaMemsetAsync(p.ready, 0, n_blobs * sizeof(int), st);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(num_sms() * per_sm);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kFusedSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return rec ? cudaLaunchKernelEx(&cfg, chunk_overlap_kernel<true>, tk, tq, tv, ty, p, n_heads)
                   : cudaLaunchKernelEx(&cfg, chunk_overlap_kernel<false>, tk, tq, tv, ty, p, n_heads);
    }
    chunk_prep_kernel<<<dim3(nchunks, s.Hv, s.B), kThreads, kP1Smem, st>>>(tk, tq, tv, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (rec) chunk_state_kernel<true><<<dim3(s.Hv, s.B), kThreads, kP2Smem, st>>>(ty, p);
    else chunk_state_kernel<false><<<dim3(s.Hv, s.B), kThreads, kP2Smem, st>>>(ty, p);
    return cudaGetLastError();
}

}  // namespace gdn
