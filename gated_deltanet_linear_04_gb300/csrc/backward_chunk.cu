// Backward pass of the recurrence in chunked (WY / UT-transform) form on the
// 5th-generation tensor cores.  Every head size of the chunked forward (Dk,
// Dv of 32, 64 or 128) runs on 128-wide tiles and records: the tiles' columns
// past the head load as zeros, so the padded rows and columns of every
// product and record are exact zeros, and the global writes are clipped to
// the head.
//
// The pages ("mlex 0.1.2, src/models/gated_delta.rs", the per-timestep loop;
// "mlx-bun 0.4.0 -> 1.0.0, package/src/model/qwen3-delta.ts",
// gated_delta_step) define the forward step; chunk_form.cuh re-blocks it into
// chunks of 64 steps.  This file differentiates those chunk products.  For a
// chunk with start state S0, G the gradient of the state at its end, and the
// forward's quantities (E[r,i] = 2^(lg_r - lg_i), gamma_r = 2^lg_r,
// F_r = 2^(lg_63 - lg_r), A, T = (I + A)^-1, D = T Z with Z = diag(beta) R,
// R = V - diag(gamma) K S0^T, P = M o Q K^T, M the lower triangle of E):
//   dD   = diag(F) K G^T + P^T dY          dZ = T^T dD        dR = diag(beta) dZ
//   G_prev = gamma_63 G + dY^T diag(gamma) Q - dR^T diag(gamma) K
//   dP   = dY D^T,  dA = -tril(dZ D^T, -1),  H = dA o beta_r E
//   dQ   = diag(gamma) dY S0 + (dP o M) K
//   dK   = diag(F) D G + (dP o M)^T Q - diag(gamma) dR S0 + (H + H^T) K
//   dV   = dR
//   dbeta = rowsum(dZ o R) + rowsum(dA o E o K K^T)
//   dlog g_t = sum_{r>=t} gamma_r dgamma_r + sum_{r<t} F_r dF_r
//              + sum_{r>=t, i<t} (dP o P + dA o A)[r,i] + gamma_63 <G, S0>
// with gamma_r dgamma_r = <dY_r, (gamma Q S0^T)_r> - beta_r <dZ_r, (gamma K S0^T)_r>,
// F_r dF_r = F_r <(D G)_r, K_r>, and dg = dlog g / g (each term of dlog g_t
// is one that log g_t scales, so no difference of prefix sums is formed).
//
// Launches, after the chunked forward has stored every chunk's start state
// S0 and D^T (the forward kernels' records):
//  1. images, one CTA per chunk: dD = Wb G^T + X1 with the state-independent
//     Wb = T^T diag(F) K and X1 = T^T P^T dY, and Cq = dY^T diag(gamma) Q,
//     written as the chain's shared-memory images;
//  2. chain, one CTA per head walking its chunks backwards with G in TMEM:
//     dZ^T = X1^T + G Wb^T, then G <- gamma_63 G + Cq + (dZ^T diag(beta))
//     (-gamma K); it stores G and dZ^T of every chunk.  When the heads take
//     at most a quarter of the SMs, 1 and 2 run as one cooperative launch
//     (the other CTAs produce the images, last chunk first, each published
//     by a ready flag that its chain acquires before loading it);
//  3. gradients I, one CTA per chunk: dv = beta dZ, gamma S0 products, dP
//     and dZ D^T, the 64 x 64 terms (dP o M, H + H^T, the dlog g staircase,
//     dbeta);
//  4. gradients II, one CTA per chunk: dQ^T and dK^T on the tensor cores
//     (M = 128 = Dk), the F dF terms and dg; dq and dk are added with
//     atomics (summed over the v-heads of a k-head).
// Every product is tf32 with f32 accumulation; every f32 operand written to
// shared memory is rounded to tf32, and the operands read from TMEM (S0, G)
// are used as tf32 by truncation, as in the forward.  Masked steps (and the
// steps past T of a last chunk) enter with g = 1, beta = 0 and dY = 0, so
// their dq, dk and dv come out exactly zero; their dg and dbeta are left at
// zero; wholly masked chunks are skipped by every launch.
#include <climits>

#include "chunk_form.cuh"
#include "common.cuh"
#include "internal.h"
#include "mask_scan.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace chunkform;

// ---- chain image (launch 1 -> 2), one per chunk
constexpr uint32_t I_WB = 0;          // Wb [64 r][128 dk] tf32, 4 K-tiles of 8 KiB (B operand)
constexpr uint32_t I_X1 = 32768;      // X1^T [128 dv][64 r] f32, thread order (chunk_form.cuh records)
constexpr uint32_t I_CQ = 65536;      // Cq [128 dv][128 dk] f32, thread order
constexpr uint32_t I_META = 131072;   // beta[64], then 2^lg_63 at +256
constexpr uint32_t I_NGK = 132096;    // (-gamma K)^T [128 dk][64 r] tf32, 2 K-tiles of 16 KiB (B operand)
constexpr uint32_t kImgA = 65536;     // Wb, X1^T: what the chain's first product reads
constexpr uint32_t kImgB = I_NGK + 32768 - kImgA;   // Cq, meta, (-gamma K)^T
constexpr size_t kImgBytes = I_NGK + 32768;
// ---- outputs of launch 3 for launch 4, in the same space, one per chunk
constexpr uint32_t O_B3 = 0;          // [dP o M ; H + H^T] [128][64] tf32, 2 K-tiles of 16 KiB
constexpr uint32_t O_DPMT = 32768;    // (dP o M)^T [64][64] tf32, 2 K-tiles of 8 KiB
constexpr uint32_t O_PART = 49152;    // 64 f32: dlog g_t without the F dF and <G, S0> terms
constexpr size_t kOutBytes = O_PART + 256;
static_assert(kOutBytes <= kImgBytes, "the second outputs reuse the image space");
static_assert(kImgA % 1024 == 0 && I_NGK % 1024 == 0 && kImgBytes % 1024 == 0, "tiles on 1 KiB boundaries");

struct BcParams {
    const float *g, *beta;
    const uint8_t *mask;
    const int *order;              // row slot -> batch row (masked batches), or null
    const float *rec_s, *rec_d;    // forward records: S0 and D^T of every chunk
    float *rec_g, *rec_z;          // chain records: G at every chunk's end, dZ^T
    uint8_t *img;                  // chain images, then launch 3's outputs
    const float *dstate_out;
    float *dq, *dk, *dv, *dg, *dbeta, *dstate_in;
    unsigned *err;
    int B, T, Hk, Hv, Dk, Dv, nchunks;
};

struct BcShared {
    uint64_t bar0, bar1, bar2;
    uint32_t tmem_slot;
    int s_word;
    float s_g[kC], s_b[kC];
    __align__(16) float s_lg[kC];
    __align__(16) float s_gam[kC];
    __align__(16) float s_beta[kC];
    __align__(16) float s_bg[kC];
    __align__(16) float s_kc[kC];
    __align__(16) float s_ok[kC];          // 1 for a valid step, 0 for a masked one or one past T
    __align__(16) float s_red[2][4][kC];   // per-TMEM-quad column sums of two quantities
    __align__(16) float s_vec[3][kC];
    float s_scalar[2];
};

__device__ __forceinline__ size_t chunk_index(const BcParams &p, int b, int hv, int c) {
    return ((size_t)b * p.Hv + hv) * p.nchunks + c;
}

// Gates of chunk c of head (b, hv) into shared memory and the step factors
// (warp 0); a masked step or one past T enters with g = 1, beta = 0,
// s_ok = 0.  Returns whether the chunk holds a valid step.  Block-wide.
__device__ __forceinline__ bool chunk_gates(const BcParams &p, BcShared &sh, int c, int b, int hv) {
    const int tid = threadIdx.x, t = c * kC + tid;
    int m = 0;
    if (tid < kC) {
        float gg = 1.0f, bb = 0.0f;
        if (t < p.T) {
            m = p.mask == nullptr ? 1 : (p.mask[(size_t)b * p.T + t] != 0);
            if (m) {
                const size_t gi = ((size_t)b * p.T + t) * p.Hv + hv;
                gg = p.g[gi];
                bb = p.beta[gi];
            }
        }
        sh.s_g[tid] = gg;
        sh.s_b[tid] = bb;
        sh.s_ok[tid] = m ? 1.0f : 0.0f;
    }
    const bool any = __syncthreads_or(m) != 0;
    if (any && (tid >> 5) == 0)
        step_factors(tid & 31, sh.s_g, sh.s_b, sh.s_lg, sh.s_gam, sh.s_kc, sh.s_beta, sh.s_bg);
    __syncthreads();
    return any;
}

// Sum over the 32 lanes of a warp of each of a lane's 32 values: value j's sum
// lands in lane j (five exchanges, each halving the vector).
__device__ __forceinline__ float transpose_sum32(float (&x)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < o; ++j) {
            const float send = up ? x[j] : x[j + o];
            const float keep = up ? x[j + o] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return x[0];
}

// Values v[j] of this thread (matrix row `row`, columns c0 + j) written as
// the transposed tf32 operand: element (tile row n0 + c0 + j, K index row) of
// a 128B-swizzled tile whose K-tiles (32 K values) are kt_bytes apart.  The
// lanes of a warp (consecutive rows) fill one 128-byte tile row per store.
template <int N>
__device__ __forceinline__ void put_transposed(uint8_t *sm, uint32_t dst, uint32_t kt_bytes, int n0, int row,
                                               const float (&v)[N], int c0) {
    const uint32_t base = dst + (uint32_t)(row >> 5) * kt_bytes;
    const uint32_t kb = (uint32_t)(row & 31) * 4u;
#pragma unroll
    for (int j = 0; j < N; ++j)
        *reinterpret_cast<float *>(sm + base + umma::sw128((uint32_t)(n0 + c0 + j), kb)) = umma::to_tf32(v[j]);
}

// (sign * scale o X)^T [128 dk][64 r] tf32 (2 K-tiles of 16 KiB) from the K
// (row_base 0) or Q (row_base 64) rows of the bf16 KQ tile; scale null = 1.
// Lanes take consecutive dk, each thread 4 consecutive r of two row quads
// (warp w: rows 4w and 4w + 32), the quad's factors loaded once.
__device__ __forceinline__ void build_xt(uint8_t *sm, uint32_t kq_off, int row_base, uint32_t dst,
                                         const float *scale, float sign, int tid) {
    const int lane = tid & 31, w = tid >> 5;
#pragma unroll
    for (int rp = 0; rp < 2; ++rp) {
        const int r = (w + 8 * rp) * 4;
        const float4 sc = scale != nullptr ? ld4(scale + r) : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
#pragma unroll
        for (int j = 0; j < kD / 32; ++j) {
            const int dk = lane + 32 * j;
            st_tf32x4(sm, dst + (r >> 5) * kSlot + umma::sw128(dk, (r & 31) * 4),
                      sign * sc.x * kq_elem(sm, kq_off, row_base + r, dk),
                      sign * sc.y * kq_elem(sm, kq_off, row_base + r + 1, dk),
                      sign * sc.z * kq_elem(sm, kq_off, row_base + r + 2, dk),
                      sign * sc.w * kq_elem(sm, kq_off, row_base + r + 3, dk));
        }
    }
}

// (scale o X)[r][dk] as tile rows dst_row + r of a tf32 operand whose K-tiles
// are kt_bytes apart, X the K (row_base 0) or Q (64) rows of the KQ tile; a
// warp covers one row r, 4 consecutive dk per lane.
__device__ __forceinline__ void build_x_rows(uint8_t *sm, uint32_t kq_off, int row_base, uint32_t dst,
                                             uint32_t kt_bytes, int dst_row, const float *scale, int tid) {
    for (int i = tid; i < kC * kD / 4; i += kThreads) {
        const int r = i >> 5, dk = (i & 31) * 4;
        const float sc = scale[r];
        const uint2 xx = *reinterpret_cast<const uint2 *>(
            sm + kq_off + (dk >> 6) * kSlot + umma::sw128(row_base + r, (dk & 63) * 2));
        st_tf32x4(sm, dst + (dk >> 5) * kt_bytes + umma::sw128(dst_row + r, (dk & 31) * 4),
                  sc * __uint_as_float(xx.x << 16), sc * __uint_as_float(xx.x & 0xffff0000u),
                  sc * __uint_as_float(xx.y << 16), sc * __uint_as_float(xx.y & 0xffff0000u));
    }
}

// dY of a valid step (else 0) from the plain bf16 [64][128] dY tile
__device__ __forceinline__ float dy_at(const uint8_t *sm, uint32_t dy_off, const float *s_ok, int r, int dv) {
    return s_ok[r] != 0.0f ? bf16_to_f32(reinterpret_cast<const uint16_t *>(sm + dy_off)[r * kD + dv]) : 0.0f;
}

// dY[r][dv] (invalid steps 0) as tile rows 0-63 of a tf32 operand whose
// K-tiles are kt_bytes apart
__device__ __forceinline__ void build_dy_rows(uint8_t *sm, uint32_t dy_off, uint32_t dst, uint32_t kt_bytes,
                                              const float *s_ok, int tid) {
    for (int i = tid; i < kC * kD / 4; i += kThreads) {
        const int r = i >> 5, dv = (i & 31) * 4;
        const bool ok = s_ok[r] != 0.0f;
        const uint2 xx = *reinterpret_cast<const uint2 *>(sm + dy_off + r * (kD * 2) + dv * 2);
        st_tf32x4(sm, dst + (dv >> 5) * kt_bytes + umma::sw128(r, (dv & 31) * 4),
                  ok ? __uint_as_float(xx.x << 16) : 0.0f, ok ? __uint_as_float(xx.x & 0xffff0000u) : 0.0f,
                  ok ? __uint_as_float(xx.y << 16) : 0.0f, ok ? __uint_as_float(xx.y & 0xffff0000u) : 0.0f);
    }
}

// dY^T [128 dv][64 r] tf32 (2 K-tiles of 16 KiB), invalid steps 0 (the
// thread layout of build_xt)
__device__ __forceinline__ void build_dyt(uint8_t *sm, uint32_t dy_off, uint32_t dst, const float *s_ok, int tid) {
    const int lane = tid & 31, w = tid >> 5;
#pragma unroll
    for (int rp = 0; rp < 2; ++rp) {
        const int r = (w + 8 * rp) * 4;
#pragma unroll
        for (int j = 0; j < kD / 32; ++j) {
            const int dv = lane + 32 * j;
            st_tf32x4(sm, dst + (r >> 5) * kSlot + umma::sw128(dv, (r & 31) * 4), dy_at(sm, dy_off, s_ok, r, dv),
                      dy_at(sm, dy_off, s_ok, r + 1, dv), dy_at(sm, dy_off, s_ok, r + 2, dv),
                      dy_at(sm, dy_off, s_ok, r + 3, dv));
        }
    }
}

// T^T as a tf32 B operand [64 r][64 i] (element (r, i) = T[i][r]), 2 K-tiles of 8 KiB
__device__ __forceinline__ void tt_tile(const float *As, uint8_t *sm, uint32_t dst, int tid) {
    for (int idx = tid; idx < kC * kC / 4; idx += kThreads) {
        const int i = idx & (kC - 1), r4 = (idx >> 6) * 4;
        const float4 t = ld4(As + aidx(i, r4));
        const uint32_t base = dst + (uint32_t)(i >> 5) * 8192u, kb = (uint32_t)(i & 31) * 4u;
        *reinterpret_cast<float *>(sm + base + umma::sw128(r4, kb)) = umma::to_tf32(t.x);
        *reinterpret_cast<float *>(sm + base + umma::sw128(r4 + 1, kb)) = umma::to_tf32(t.y);
        *reinterpret_cast<float *>(sm + base + umma::sw128(r4 + 2, kb)) = umma::to_tf32(t.z);
        *reinterpret_cast<float *>(sm + base + umma::sw128(r4 + 3, kb)) = umma::to_tf32(t.w);
    }
}

// thread's 64 columns of a [128][128] record, 32 of a [128][64] one
__device__ __forceinline__ void load_rec128(const float *rec, int row, int half, float (&v)[64]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float4 x = *rec128_at(rec, row, half, j);
        v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
    }
}
__device__ __forceinline__ void load_rec64(const float *rec, int row, int half, float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 x = *rec64_at(rec, row, half, j);
        v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
    }
}

// 64 values into TMEM columns [col, col + 64) of this thread's lane
__device__ __forceinline__ void tmem_put64(uint32_t taddr, const float (&v)[64]) {
    float a[32], b[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        a[j] = v[j];
        b[j] = v[32 + j];
    }
    umma::tmem_st32(taddr, a);
    umma::tmem_st32(taddr + 32, b);
}

// The k, q (128B-swizzled halves, K rows 0-63 / Q rows 64-127) and one
// plain [64][128] bf16 tile (v or dY) of chunk rows starting at `rowg`, all
// counted on `bar`, whose single arrival (with the expected bytes) the caller
// makes once for everything that phase loads.
constexpr uint32_t kKQVBytes = 4 * 8192 + 16384;

// A plain [64][128] bf16 tile (v or dY) of head hx, in the map form of the
// head size (chunk_form.cuh: 2-D at Dv = 128, else the padded 3-D form whose
// columns past the head read as zeros).
__device__ __forceinline__ void issue_x_tile(uint8_t *dst, const CUtensorMap *tm_x, int Dv, int hx, int rowg,
                                             uint64_t *bar) {
    if (Dv == kD) tma_load_2d(dst, tm_x, hx * kD, rowg, bar);
    else tma_load_3d(dst, tm_x, 0, hx, rowg, bar);
}

__device__ __forceinline__ void issue_kq_tile(uint8_t *sm, uint32_t kq_off, uint32_t x_off, const CUtensorMap *tm_k,
                                              const CUtensorMap *tm_q, const CUtensorMap *tm_x, int Dk, int Dv,
                                              int hk, int hx, int rowg, uint64_t *bar) {
    if (Dk == kD) {
        tma_load_2d(sm + kq_off, tm_k, hk * kD, rowg, bar);
        tma_load_2d(sm + kq_off + kSlot, tm_k, hk * kD + 64, rowg, bar);
        tma_load_2d(sm + kq_off + 8192, tm_q, hk * kD, rowg, bar);
        tma_load_2d(sm + kq_off + kSlot + 8192, tm_q, hk * kD + 64, rowg, bar);
    } else {
        tma_load_3d(sm + kq_off, tm_k, 0, hk, rowg, bar);
        tma_load_3d(sm + kq_off + kSlot, tm_k, 64, hk, rowg, bar);
        tma_load_3d(sm + kq_off + 8192, tm_q, 0, hk, rowg, bar);
        tma_load_3d(sm + kq_off + kSlot + 8192, tm_q, 64, hk, rowg, bar);
    }
    issue_x_tile(sm + x_off, tm_x, Dv, hx, rowg, bar);
}

// barriers and TMEM of a CTA; returns the TMEM base
__device__ __forceinline__ uint32_t bc_setup(BcShared &sh, uint32_t cols) {
    if (threadIdx.x == 0) {
        mbar_init(&sh.bar0, 1);
        mbar_init(&sh.bar1, 1);
        mbar_init(&sh.bar2, 1);
        fence_mbar_init();
    }
    if ((threadIdx.x >> 5) == 0) {
        umma::tmem_alloc(&sh.tmem_slot, cols);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    return sh.tmem_slot;
}

__device__ __forceinline__ void bc_teardown(uint32_t tmem, uint32_t cols) {
    umma::fence_before_sync();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) umma::tmem_dealloc(tmem, cols);
}

__device__ __forceinline__ uint8_t *aligned_smem(uint8_t *raw, uint32_t &base) {
    base = (smem_u32(raw) + 1023u) & ~1023u;
    return raw + (base - smem_u32(raw));
}

// generic smem writes and TMEM stores visible to the next MMA issue
__device__ __forceinline__ void publish_operands() {
    fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
}

// bounded wait on an mbarrier phase by every thread, agreed across the CTA
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity, unsigned *err) {
    const bool w = __syncthreads_and(mbar_wait(bar, parity, err)) != 0;
    umma::fence_after_sync();
    return w;
}

// ===========================================================================
// launch 1: chain images, one CTA per (chunk, hv, b)
// ===========================================================================
constexpr uint32_t L_KQ = 0 * kSlot;    // K / Q (bf16, TMA); then T^T [64 r][64 i] tf32
constexpr uint32_t L_DY = 2 * kSlot;    // dY plain bf16 (TMA); then the inverse's scratch
constexpr uint32_t L_KT = 3 * kSlot;    // (F K)^T [128][64]; then Wb [64 r][128 dk]
constexpr uint32_t L_NGK = 5 * kSlot;   // (-gamma K)^T [128][64]
constexpr uint32_t L_DYT = 7 * kSlot;   // dY^T [128 dv][64 i]; then Z1 = dY^T P as an A operand
constexpr uint32_t L_GQT = 9 * kSlot;   // (gamma Q)^T [128 dk][64 i]
constexpr uint32_t L_PT = 11 * kSlot;   // P^T [64 r][64 i] (element (r, i) = P[i][r]), 2 K-tiles of 8 KiB
constexpr uint32_t L_A = 12 * kSlot;    // A, then T, plain f32 [64][64]
constexpr uint32_t L_CQS = 9 * kSlot;   // Cq staged for its bulk store (slots 9-12, dead by then)
constexpr uint32_t L_META = L_DY + 8192;   // beta and 2^lg_63 staged (past the inverse's 4 KiB scratch)
constexpr uint32_t kLSmem = 13 * kSlot + 1024;
// TMEM: QK 0-63 (then X1^T), Z1 64-127, Wb^T 128-191, Cq 256-383
constexpr uint32_t L_CQK = 0, L_CZ1 = 64, L_CWB = 128, L_CCQ = 256;

// One chain image: chunk c of head (b, hv), whose gates and step factors
// chunk_gates has put in shared memory; the TMA and MMA barrier phases carry
// over from unit to unit.  Every byte of the image leaves by bulk stores from
// shared memory (Wb and (-gamma K)^T as operand tiles, Cq, X1^T and the meta
// staged in the thread order of the chain), committed and waited for before
// returning, so the image is complete in memory when this returns true.
__device__ __forceinline__ bool image_unit(const BcParams &p, const CUtensorMap *tm_k, const CUtensorMap *tm_q,
                                           const CUtensorMap *tm_dy, BcShared &sh, uint8_t *sm, uint32_t base,
                                           uint32_t tmem, int c, int b, int hv, uint32_t &tma_phase,
                                           uint32_t &mma_phase) {
    const int tid = threadIdx.x, warp = tid >> 5;
    const int quad = warp & 3, half = warp >> 2, row = quad * 32 + (tid & 31);
    const int hk = hv / (p.Hv / p.Hk);
    const uint32_t lt = tmem + ((uint32_t)(quad * 32) << 16);
    float *As = reinterpret_cast<float *>(sm + L_A);
    float *Ys = reinterpret_cast<float *>(sm + L_DY);
    uint8_t *img = p.img + chunk_index(p, b, hv, c) * kImgBytes;

    if (tid == 0) {
        mbar_expect_tx(&sh.bar0, kKQVBytes);
        issue_kq_tile(sm, L_KQ, L_DY, tm_k, tm_q, tm_dy, p.Dk, p.Dv, hk, hv, b * p.T + c * kC, &sh.bar0);
    }
    bool ok = wait_all(&sh.bar0, tma_phase++ & 1u, p.err);
    if (ok) {
        if (tid == 0) {
            issue_kq(tmem, base, L_KQ);
            umma::mma_commit(&sh.bar2);
        }
        build_xt(sm, L_KQ, 0, L_KT, sh.s_kc, 1.0f, tid);
        build_xt(sm, L_KQ, 0, L_NGK, sh.s_gam, -1.0f, tid);
        build_xt(sm, L_KQ, 64, L_GQT, sh.s_gam, 1.0f, tid);
        build_dyt(sm, L_DY, L_DYT, sh.s_ok, tid);
        ok = wait_all(&sh.bar2, mma_phase++ & 1u, p.err);
    }
    if (ok) {
        // A from K K^T (quads 0-1); P^T from Q K^T (quads 2-3)
        if (quad < 2) {
            build_a(lt + L_CQK, As, sh.s_lg, sh.s_beta, row, half);
        } else {
            float qk[32], pv[32];
            umma::tmem_ld32(lt + L_CQK + half * 32, qk);
            umma::tmem_ld_wait();
            const int i = row - 64;
            const float li = sh.s_lg[i];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = half * 32 + j;
                pv[j] = r <= i ? decay(li - sh.s_lg[r]) * qk[j] : 0.0f;
            }
            put_transposed<32>(sm, L_PT, 8192, 0, i, pv, half * 32);
        }
        umma::fence_before_sync();
        __syncthreads();
        invert_unit_lower(As, Ys, tid);
        tt_tile(As, sm, L_KQ, tid);
        publish_operands();
        if (tid == 0) {
            const uint32_t id64 = umma::idesc(128, 64, umma::kFmtTF32), id128 = umma::idesc(128, 128, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t kt = k >> 2, ko = (k & 3) * 32;
                const uint64_t tt = umma::desc_sw128(base + L_KQ + kt * 8192 + ko);
                const uint64_t dyt = umma::desc_sw128(base + L_DYT + kt * kSlot + ko);
                // Wb^T = (F K)^T T ; Z1 = dY^T P ; Cq = dY^T (gamma Q)
                umma::mma_tf32(tmem + L_CWB, umma::desc_sw128(base + L_KT + kt * kSlot + ko), tt, id64, k > 0);
                umma::mma_tf32(tmem + L_CZ1, dyt, umma::desc_sw128(base + L_PT + kt * 8192 + ko), id64, k > 0);
                umma::mma_tf32(tmem + L_CCQ, dyt, umma::desc_sw128(base + L_GQT + kt * kSlot + ko), id128, k > 0);
            }
            umma::mma_commit(&sh.bar2);
        }
        ok = wait_all(&sh.bar2, mma_phase++ & 1u, p.err);
    }
    if (ok) {
        {
            float z1[32], wb[32];
            umma::tmem_ld32(lt + L_CZ1 + half * 32, z1);
            umma::tmem_ld32(lt + L_CWB + half * 32, wb);
            umma::tmem_ld_wait();
            dt_tile(z1, sm, L_DYT, row, half);                        // Z1 [dv][i] as an A operand
            put_transposed<32>(sm, L_KT, 8192, 0, row, wb, half * 32);  // Wb [r][dk]
        }
        {
            // Cq, in the chain's thread order, into the dead (gamma Q)^T, P^T and A slots
            float ca[32], cb[32];
            umma::tmem_ld32(lt + L_CCQ + half * 64, ca);
            umma::tmem_ld32(lt + L_CCQ + half * 64 + 32, cb);
            umma::tmem_ld_wait();
            float *cq = reinterpret_cast<float *>(sm + L_CQS);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                *rec128_at(cq, row, half, j) = make_float4(ca[4 * j], ca[4 * j + 1], ca[4 * j + 2], ca[4 * j + 3]);
                *rec128_at(cq, row, half, 8 + j) = make_float4(cb[4 * j], cb[4 * j + 1], cb[4 * j + 2], cb[4 * j + 3]);
            }
        }
        float *meta = reinterpret_cast<float *>(sm + L_META);
        if (tid < kC) meta[tid] = sh.s_beta[tid];
        if (tid == 0) meta[64] = sh.s_gam[kC - 1];
        publish_operands();
        if (tid == 0) {
            // X1^T = Z1 T (into the dead QK columns)
            const uint32_t id64 = umma::idesc(128, 64, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t kt = k >> 2, ko = (k & 3) * 32;
                umma::mma_tf32(tmem + L_CQK, umma::desc_sw128(base + L_DYT + kt * kSlot + ko),
                               umma::desc_sw128(base + L_KQ + kt * 8192 + ko), id64, k > 0);
            }
            umma::mma_commit(&sh.bar2);
            bulk_store(img + I_WB, sm + L_KT, 32768);
            bulk_store(img + I_NGK, sm + L_NGK, 32768);
            bulk_store(img + I_CQ, sm + L_CQS, 65536);
            bulk_store(img + I_META, sm + L_META, 512);
        }
        ok = wait_all(&sh.bar2, mma_phase++ & 1u, p.err);
    }
    if (ok) {
        // X1^T into the Z1 tile's slots (the product that read them is done)
        float x1[32];
        umma::tmem_ld32(lt + L_CQK + half * 32, x1);
        umma::tmem_ld_wait();
        store_rec64(reinterpret_cast<float *>(sm + L_DYT), row, half, x1);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) bulk_store(img + I_X1, sm + L_DYT, 32768);
    } else if (tid == 0) {
        mbar_wait(&sh.bar2, mma_phase & 1u, nullptr);   // give in-flight MMAs a bounded chance to drain
    }
    if (tid == 0) {
        bulk_commit();
        bulk_wait_all();   // the image is in memory (and shared memory free for the next unit)
    }
    umma::fence_before_sync();
    __syncthreads();
    return ok;
}

__global__ void __launch_bounds__(kThreads, 1) bc_image_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                const __grid_constant__ CUtensorMap tm_q,
                                                                const __grid_constant__ CUtensorMap tm_dy,
                                                                const BcParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ BcShared sh;
    uint32_t base;
    uint8_t *sm = aligned_smem(smem_raw, base);
    const int c = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
    if (!chunk_gates(p, sh, c, b, hv)) return;
    const uint32_t tmem = bc_setup(sh, 512);
    uint32_t tma_phase = 0, mma_phase = 0;
    image_unit(p, &tm_k, &tm_q, &tm_dy, sh, sm, base, tmem, c, b, hv, tma_phase, mma_phase);
    bc_teardown(tmem, 512);
}

// ===========================================================================
// launch 2: the reverse chain, one CTA per (hv, row slot)
// ===========================================================================
constexpr uint32_t R_DZB = (uint32_t)kImgBytes;   // dZ^T diag(beta) [128 dv][64 r] tf32 (A operand), 32 KiB
constexpr uint32_t kRSmem = R_DZB + 32768 + 1024;
constexpr uint32_t R_CG = 0, R_CZ = 128;          // TMEM: G (128 columns), dZ^T (64)

// Largest chunk index <= from holding a valid step of mask row `mrow`, or -1.  Block-wide.
__device__ __forceinline__ int prev_active(const uint8_t *mrow, int T, int from, int *s_word) {
    if (mrow == nullptr) return from;
    while (from >= 0) {
        const int ch = from - (int)threadIdx.x;
        const bool any = ch >= 0 && chunk_has_valid(mrow, T, ch);
        if (threadIdx.x == 0) *s_word = INT_MAX;
        __syncthreads();
        if (any) atomicMin(s_word, (int)threadIdx.x);
        __syncthreads();
        const int w = *s_word;
        __syncthreads();
        if (w != INT_MAX) return from - w;
        from -= (int)blockDim.x;
    }
    return -1;
}

// Bounded wait (acquire) for a chunk image's ready flag, then order it
// before the async-proxy bulk loads that read the image.
__device__ __forceinline__ bool wait_image(const int *flag, unsigned *err) {
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

// Publishes an image whose bulk stores this thread has seen complete.
__device__ __forceinline__ void publish_image(int *flag) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}

// The reverse chain of head (b, hv).  With `ready` (overlapped form), each
// chunk's image is waited for by its flag before it is loaded; after one
// wait has given up no further one is made.
__device__ __forceinline__ void chain_head(const BcParams &p, BcShared &sh, uint8_t *sm, uint32_t base,
                                           uint32_t tmem, int b, int hv, const int *ready) {
    const int tid = threadIdx.x, warp = tid >> 5;
    const int quad = warp & 3, half = warp >> 2, row = quad * 32 + (tid & 31);
    const int T = p.T;
    const uint32_t lt = tmem + ((uint32_t)(quad * 32) << 16);
    bool flag_gave_up = false;   // thread 0
    const uint8_t *mrow = p.mask == nullptr ? nullptr : p.mask + (size_t)b * T;

    // G = the gradient of the final state -> TMEM
    state_to_tmem(p.dstate_out, lt + R_CG, b, hv, p.Hv, p.Dk, p.Dv, row, half);

    bool a_pending = false, b_pending = false;   // thread 0: copies in flight
    uint32_t a_par = 0, b_par = 0;
    auto load_a = [&](int ch, int it) {
        if (tid == 0) {
            if (ready != nullptr && !flag_gave_up)
                flag_gave_up = !wait_image(ready + chunk_index(p, b, hv, ch), p.err);
            mbar_expect_tx(&sh.bar0, kImgA);
            bulk_load(sm, p.img + chunk_index(p, b, hv, ch) * kImgBytes, kImgA, &sh.bar0);
            a_pending = true;
            a_par = (uint32_t)(it & 1);
        }
    };
    auto load_b = [&](int ch, int it) {
        if (tid == 0) {
            mbar_expect_tx(&sh.bar1, kImgB);
            bulk_load(sm + kImgA, p.img + chunk_index(p, b, hv, ch) * kImgBytes + kImgA, kImgB, &sh.bar1);
            b_pending = true;
            b_par = (uint32_t)(it & 1);
        }
    };

    int c = prev_active(mrow, T, p.nchunks - 1, &sh.s_word);
    if (c >= 0) {
        load_a(c, 0);
        load_b(c, 0);
    }
    umma::fence_before_sync();
    __syncthreads();
    uint32_t mma_phase = 0;
    bool ok = true;
    for (int it = 0; c >= 0 && ok; ++it) {
        const size_t ci = chunk_index(p, b, hv, c);
        if (!wait_all(&sh.bar0, (uint32_t)(it & 1), p.err)) { ok = false; break; }
        if (tid == 0) a_pending = false;
        // X1^T -> the dZ^T accumulator
        {
            float x1[32];
            load_rec64(reinterpret_cast<const float *>(sm + I_X1), row, half, x1);
            umma::tmem_st32(lt + R_CZ + half * 32, x1);
            umma::tmem_st_wait();
        }
        publish_operands();
        if (tid == 0) {
            // dZ^T += G Wb^T, G read from TMEM
            const uint32_t id = umma::idesc(128, 64, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                umma::mma_tf32_tmem_a(tmem + R_CZ, tmem + R_CG + 8 * k,
                                      umma::desc_sw128(base + I_WB + (k >> 2) * 8192 + (k & 3) * 32), id, true);
            umma::mma_commit(&sh.bar2);
        }
        // G (the gradient at this chunk's end) -> its record, meanwhile
        float gv[64];
        {
            float ga[32], gb[32];
            umma::tmem_ld32(lt + R_CG + half * 64, ga);
            umma::tmem_ld32(lt + R_CG + half * 64 + 32, gb);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                gv[j] = ga[j];
                gv[32 + j] = gb[j];
            }
            float *rg = p.rec_g + ci * kRec128;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                *rec128_at(rg, row, half, j) = make_float4(gv[4 * j], gv[4 * j + 1], gv[4 * j + 2], gv[4 * j + 3]);
        }
        const int cn = prev_active(mrow, T, c - 1, &sh.s_word);
        if (!wait_all(&sh.bar2, mma_phase++ & 1u, p.err)) { ok = false; break; }
        if (cn >= 0) load_a(cn, it + 1);   // Wb and X1^T have been consumed
        if (!wait_all(&sh.bar1, (uint32_t)(it & 1), p.err)) { ok = false; break; }
        if (tid == 0) b_pending = false;
        const float* meta = reinterpret_cast<const float *>(sm + I_META);
        const float gl = meta[64];
        // G <- 2^lg_63 G + Cq
        {
            const float *cq = reinterpret_cast<const float *>(sm + I_CQ);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float4 x = *rec128_at(cq, row, half, j);
                gv[4 * j] = fmaf(gl, gv[4 * j], x.x);
                gv[4 * j + 1] = fmaf(gl, gv[4 * j + 1], x.y);
                gv[4 * j + 2] = fmaf(gl, gv[4 * j + 2], x.z);
                gv[4 * j + 3] = fmaf(gl, gv[4 * j + 3], x.w);
            }
            tmem_put64(lt + R_CG + half * 64, gv);
        }
        // dZ^T: its record, and dZ^T diag(beta) as the A operand (dv = beta dZ
        // is written by the first gradient pass, off the chain)
        {
            float z[32];
            umma::tmem_ld32(lt + R_CZ + half * 32, z);
            umma::tmem_ld_wait();
            store_rec64(p.rec_z + ci * kRec64, row, half, z);
#pragma unroll
            for (int j = 0; j < 32; ++j) z[j] *= meta[half * 32 + j];
            dt_tile(z, sm, R_DZB, row, half);
        }
        umma::tmem_st_wait();
        publish_operands();
        if (tid == 0) {
            // G += (dZ^T diag(beta)) (-gamma K)
            const uint32_t id = umma::idesc(128, 128, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t kt = k >> 2, ko = (k & 3) * 32;
                umma::mma_tf32(tmem + R_CG, umma::desc_sw128(base + R_DZB + kt * kSlot + ko),
                               umma::desc_sw128(base + I_NGK + kt * kSlot + ko), id, true);
            }
            umma::mma_commit(&sh.bar2);
        }
        if (!wait_all(&sh.bar2, mma_phase++ & 1u, p.err)) { ok = false; break; }
        if (cn >= 0) load_b(cn, it + 1);   // Cq, meta and (-gamma K)^T have been consumed
        c = cn;
    }
    if (__syncthreads_and(ok)) {
        state_from_tmem(p.dstate_in, lt + R_CG, b, hv, p.Hv, p.Dk, p.Dv, row, half);
    } else if (tid == 0) {
        // a wait gave up: give in-flight MMAs and copies a bounded chance to drain
        mbar_wait(&sh.bar2, mma_phase & 1u, nullptr);
        if (a_pending) mbar_wait(&sh.bar0, a_par, nullptr);
        if (b_pending) mbar_wait(&sh.bar1, b_par, nullptr);
    }
}

__global__ void __launch_bounds__(kThreads, 1) bc_chain_kernel(const BcParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ BcShared sh;
    uint32_t base;
    uint8_t *sm = aligned_smem(smem_raw, base);
    const int b = p.order != nullptr ? p.order[blockIdx.y] : (int)blockIdx.y;
    const uint32_t tmem = bc_setup(sh, 256);
    chain_head(p, sh, sm, base, tmem, b, blockIdx.x, nullptr);
    bc_teardown(tmem, 256);
}

// Overlapped form of launches 1 and 2 (cooperative, all CTAs resident): CTAs
// [0, n_heads) run the reverse chains, the others produce the chain images
// from the last chunk backwards (unit u: chunk nchunks - 1 - u / n_heads of
// head u % n_heads, in steps of the producer count), publishing each with a
// ready flag once its bulk stores are complete.
__global__ void __launch_bounds__(kThreads, 1) bc_overlap_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                  const __grid_constant__ CUtensorMap tm_q,
                                                                  const __grid_constant__ CUtensorMap tm_dy,
                                                                  const BcParams p, const int n_heads, int *ready) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ BcShared sh;
    uint32_t base;
    uint8_t *sm = aligned_smem(smem_raw, base);
    const bool is_chain = (int)blockIdx.x < n_heads;
    const uint32_t cols = is_chain ? 256u : 512u;
    const uint32_t tmem = bc_setup(sh, cols);
    if (is_chain) {
        const int slot = blockIdx.x / p.Hv, hv = blockIdx.x % p.Hv;
        const int b = p.order != nullptr ? p.order[slot] : slot;
        chain_head(p, sh, sm, base, tmem, b, hv, ready);
    } else {
        const int n_prep = (int)gridDim.x - n_heads;
        const long n_units = (long)p.nchunks * n_heads;
        uint32_t tma_phase = 0, mma_phase = 0;
        for (long u = (long)blockIdx.x - n_heads; u < n_units; u += n_prep) {
            const int c = p.nchunks - 1 - (int)(u / n_heads), h = (int)(u % n_heads);
            const int slot = h / p.Hv, hv = h % p.Hv;
            const int b = p.order != nullptr ? p.order[slot] : slot;
            if (!chunk_gates(p, sh, c, b, hv)) continue;   // the chain skips it too
            if (!image_unit(p, &tm_k, &tm_q, &tm_dy, sh, sm, base, tmem, c, b, hv, tma_phase, mma_phase)) break;
            if (threadIdx.x == 0) publish_image(ready + chunk_index(p, b, hv, c));
        }
    }
    bc_teardown(tmem, cols);
}

// ===========================================================================
// launch 3: gradients I, one CTA per (chunk, hv, b)
// ===========================================================================
constexpr uint32_t A_KQ = 0 * kSlot;    // K / Q (TMA); then D [64 i][128 dv] tf32 (4 K-tiles of 8 KiB)
constexpr uint32_t A_V = 2 * kSlot;     // V plain bf16 (TMA)
constexpr uint32_t A_DY = 3 * kSlot;    // dY plain bf16 (TMA)
constexpr uint32_t A_GKQ = 4 * kSlot;   // [gamma K ; gamma Q] [128][128] tf32 (4 K-tiles of 16 KiB);
                                        // then [dY ; dZ] [128][128]; then B3 (slots 4-5), (dP o M)^T (6), H (7)
constexpr uint32_t A_B3 = 4 * kSlot, A_DPMT = 6 * kSlot, A_H = 7 * kSlot;
constexpr uint32_t A_EKK = 8 * kSlot;   // E o K K^T plain [64][64]; then dA o A
constexpr uint32_t A_P = 9 * kSlot;     // P plain [64][64]
constexpr uint32_t A_X = 10 * kSlot;    // dP o P plain [64][64]; then its row prefix sums
constexpr uint32_t kASmem = 11 * kSlot + 1024;
// TMEM: QK 0-63 (then [dP ; dZ D^T]), [YK^T | YQ^T] 128-255, S0 256-383
constexpr uint32_t A_CQK = 0, A_CYK = 128, A_CYQ = 192, A_CS0 = 256;

__global__ void __launch_bounds__(kThreads, 1) bc_grad1_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                const __grid_constant__ CUtensorMap tm_q,
                                                                const __grid_constant__ CUtensorMap tm_v,
                                                                const __grid_constant__ CUtensorMap tm_dy,
                                                                const BcParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ BcShared sh;
    uint32_t base;
    uint8_t *sm = aligned_smem(smem_raw, base);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2, row = quad * 32 + lane;
    const int c = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
    const int hk = hv / (p.Hv / p.Hk);
    const int T = p.T, t0 = c * kC;
    if (!chunk_gates(p, sh, c, b, hv)) return;
    const uint32_t tmem = bc_setup(sh, 512);
    const uint32_t lt = tmem + ((uint32_t)(quad * 32) << 16);
    const size_t ci = chunk_index(p, b, hv, c);
    float *EKK = reinterpret_cast<float *>(sm + A_EKK);
    float *Pm = reinterpret_cast<float *>(sm + A_P);
    float *Xa = reinterpret_cast<float *>(sm + A_X);
    float *Hm = reinterpret_cast<float *>(sm + A_H);

    if (tid == 0) {
        // one arrival for the phase, with every byte it brings in
        mbar_expect_tx(&sh.bar0, kKQVBytes + 16384);
        issue_kq_tile(sm, A_KQ, A_V, &tm_k, &tm_q, &tm_v, p.Dk, p.Dv, hk, hv, b * T + t0, &sh.bar0);
        issue_x_tile(sm + A_DY, &tm_dy, p.Dv, hv, b * T + t0, &sh.bar0);
    }
    if (tid < kC) {
        sh.s_vec[0][tid] = 0.0f;   // dbeta of the dA term
    }
    // S0 -> TMEM; the dZ^T and D^T records are fetched now and used after the first products
    float z[32], dl[32];   // dZ^T[dv = row][r = 32 half + j], D^T likewise
    {
        float s0[64];
        load_rec128(p.rec_s + ci * kRec128, row, half, s0);
        load_rec64(p.rec_z + ci * kRec64, row, half, z);
        load_dt_record(p.rec_d + ci * kRec64, row, half, dl);
        tmem_put64(lt + A_CS0 + half * 64, s0);
        umma::tmem_st_wait();
    }
    uint32_t mma_phase = 0;
    bool ok = wait_all(&sh.bar0, 0, p.err);
    if (ok) {
        build_x_rows(sm, A_KQ, 0, A_GKQ, 16384, 0, sh.s_gam, tid);    // gamma K
        build_x_rows(sm, A_KQ, 64, A_GKQ, 16384, 64, sh.s_gam, tid);  // gamma Q
        publish_operands();
        if (tid == 0) {
            issue_kq(tmem, base, A_KQ);
            // [YK^T | YQ^T] = S0 [gamma K ; gamma Q]^T, S0 read from TMEM
            const uint32_t id = umma::idesc(128, 128, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                umma::mma_tf32_tmem_a(tmem + A_CYK, tmem + A_CS0 + 8 * k,
                                      umma::desc_sw128(base + A_GKQ + (k >> 2) * 16384 + (k & 3) * 32), id, k > 0);
            umma::mma_commit(&sh.bar2);
        }
        ok = wait_all(&sh.bar2, mma_phase++ & 1u, p.err);
    }
    if (ok) {
        // E o K K^T (quads 0-1) and P (quads 2-3), plain
        {
            float x[32];
            umma::tmem_ld32(lt + A_CQK + half * 32, x);
            umma::tmem_ld_wait();
            const int r = row & (kC - 1);
            const float lr = sh.s_lg[r];
            float *dst = quad < 2 ? EKK : Pm;
            const int lim = quad < 2 ? r : r + 1;   // strictly lower / lower with the diagonal
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float v4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = half * 32 + j + e;
                    v4[e] = i < lim ? decay(lr - sh.s_lg[i]) * x[j + e] : 0.0f;
                }
                st4(dst + aidx(r, half * 32 + j), make_float4(v4[0], v4[1], v4[2], v4[3]));
            }
        }
        // [dY ; dZ] as the A operand (the [gamma K ; gamma Q] tiles are dead), D as B
        put_transposed<32>(sm, A_GKQ, 16384, 64, row, z, half * 32);
        put_transposed<32>(sm, A_KQ, 8192, 0, row, dl, half * 32);
        // dv = beta dZ (a warp's 32 threads write 128 contiguous bytes per step)
        if (row < p.Dv) {
            float *dv0 = p.dv + (((size_t)b * T + t0) * p.Hv + hv) * p.Dv + row;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = half * 32 + j;
                if (t0 + r < T) dv0[(size_t)r * p.Hv * p.Dv] = sh.s_beta[r] * z[j];
            }
        }
        build_dy_rows(sm, A_DY, A_GKQ, 16384, sh.s_ok, tid);
        publish_operands();
        if (tid == 0) {
            // [dP ; dZ D^T] = [dY ; dZ] D^T
            const uint32_t id = umma::idesc(128, 64, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                umma::mma_tf32(tmem + A_CQK, umma::desc_sw128(base + A_GKQ + (k >> 2) * 16384 + (k & 3) * 32),
                               umma::desc_sw128(base + A_KQ + (k >> 2) * 8192 + (k & 3) * 32), id, k > 0);
            umma::mma_commit(&sh.bar2);
        }
        // meanwhile: gamma_r dgamma_r and the dZ o R part of dbeta, summed over dv
        {
            float yk[32], yq[32], ag[32], db[32];
            umma::tmem_ld32(lt + A_CYK + half * 32, yk);
            umma::tmem_ld32(lt + A_CYQ + half * 32, yq);
            umma::tmem_ld_wait();
            const uint16_t *Vs = reinterpret_cast<const uint16_t *>(sm + A_V);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = half * 32 + j;
                const float dyv = dy_at(sm, A_DY, sh.s_ok, r, row);
                ag[j] = dyv * yq[j] - sh.s_beta[r] * (z[j] * yk[j]);
                db[j] = z[j] * (bf16_to_f32(Vs[r * kD + row]) - yk[j]);
            }
            const float sa = transpose_sum32(ag);
            const float sd = transpose_sum32(db);
            sh.s_red[0][quad][half * 32 + lane] = sa;
            sh.s_red[1][quad][half * 32 + lane] = sd;
        }
        ok = wait_all(&sh.bar2, mma_phase++ & 1u, p.err);
    }
    if (ok) {
        // per step: gamma_r dgamma_r (s_vec[1]) and the dZ o R part of dbeta (s_vec[2])
        if (tid < kC) {
            sh.s_vec[1][tid] = (sh.s_red[0][0][tid] + sh.s_red[0][1][tid]) + (sh.s_red[0][2][tid] + sh.s_red[0][3][tid]);
            sh.s_vec[2][tid] = (sh.s_red[1][0][tid] + sh.s_red[1][1][tid]) + (sh.s_red[1][2][tid] + sh.s_red[1][3][tid]);
        }
        // the [dY ; dZ] and D tiles are dead: B3, (dP o M)^T and H take their place
        float x[32];
        umma::tmem_ld32(lt + A_CQK + half * 32, x);
        umma::tmem_ld_wait();
        if (quad < 2) {
            // dP row r: dP o M into B3 rows 0-63 and its transpose; dP o P
            const int r = row;
            const float lr = sh.s_lg[r];
            float dpm[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const int i0 = half * 32 + j;
                const float4 pp = ld4(Pm + aidx(r, i0));
                const float pv[4] = {pp.x, pp.y, pp.z, pp.w};
                float xp[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = i0 + e;
                    dpm[j + e] = i <= r ? x[j + e] * decay(lr - sh.s_lg[i]) : 0.0f;
                    xp[e] = x[j + e] * pv[e];
                }
                st4(Xa + aidx(r, i0), make_float4(xp[0], xp[1], xp[2], xp[3]));
            }
            dt_tile(dpm, sm, A_B3, r, half);
            put_transposed<32>(sm, A_DPMT, 8192, 0, r, dpm, half * 32);
        } else {
            // (dZ D^T) row r: dA = -(strictly lower part); H = dA o beta_r E; dA o A; dbeta's dA term
            const int r = row - 64;
            const float lr = sh.s_lg[r], br = sh.s_beta[r];
            float dbp = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const int i0 = half * 32 + j;
                const float4 ek = ld4(EKK + aidx(r, i0));
                const float ekv[4] = {ek.x, ek.y, ek.z, ek.w};
                float h4[4], xa[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = i0 + e;
                    const float dA = i < r ? -x[j + e] : 0.0f;
                    dbp = fmaf(dA, ekv[e], dbp);
                    h4[e] = i < r ? dA * br * decay(lr - sh.s_lg[i]) : 0.0f;
                    xa[e] = dA * (br * ekv[e]);
                }
                st4(Hm + aidx(r, i0), make_float4(h4[0], h4[1], h4[2], h4[3]));
                st4(EKK + aidx(r, i0), make_float4(xa[0], xa[1], xa[2], xa[3]));
            }
            atomicAdd(&sh.s_vec[0][r], dbp);
        }
        __syncthreads();
        if (quad >= 2) {
            // B3 rows 64-127: H + H^T
            const int r = row - 64;
            float hh[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int i = half * 32 + j;
                hh[j] = Hm[aidx(r, i)] + Hm[aidx(i, r)];
            }
            dt_tile(hh, sm, A_B3, row, half);
        }
        // row prefix sums of X = dP o P + dA o A over i < r, four threads per
        // row of 16 columns each: Xa[r][t] <- sum_{i<t} X[r][i]
        {
            const int r = tid >> 2, q = tid & 3;
            float v[16], run = 0.0f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int i = 16 * q + e;
                v[e] = i < r ? Xa[aidx(r, i)] + EKK[aidx(r, i)] : 0.0f;
                run += v[e];
            }
            // the preceding groups' total, taken from the previous lane's
            // inclusive sum: never formed by a subtraction, which would lose a
            // tiny prefix next to a large group (gates near 1e-16 make the
            // terms of one step's dlog g that small)
            float incl = run;
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, incl, o, 4);
                if (q >= o) incl += n;
            }
            const float prev = __shfl_up_sync(0xffffffffu, incl, 1, 4);
            float acc = q == 0 ? 0.0f : prev;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                Xa[aidx(r, 16 * q + e)] = acc;
                acc += v[e];
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        uint8_t *out = p.img + ci * kImgBytes;
        if (tid == 0) {
            bulk_store(out + O_B3, sm + A_B3, 32768);
            bulk_store(out + O_DPMT, sm + A_DPMT, 16384);
            bulk_commit();
        }
        // column sums over r >= t of the prefix sums (the staircase sum_{r>=t,
        // i<t} X[r][i]) and of gamma_r dgamma_r, four threads per step t
        {
            const int t = tid & (kC - 1), q = tid >> 6;
            float sx = 0.0f, sa = 0.0f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int r = 16 * q + e;
                if (r >= t) {
                    sx += Xa[aidx(r, t)];
                    sa += sh.s_vec[1][r];
                }
            }
            sh.s_red[0][q][t] = sx;
            sh.s_red[1][q][t] = sa;
        }
        __syncthreads();
        if (tid < kC) {
            const int t = tid;
            const float sx = (sh.s_red[0][0][t] + sh.s_red[0][1][t]) + (sh.s_red[0][2][t] + sh.s_red[0][3][t]);
            const float sa = (sh.s_red[1][0][t] + sh.s_red[1][1][t]) + (sh.s_red[1][2][t] + sh.s_red[1][3][t]);
            reinterpret_cast<float *>(out + O_PART)[t] = sa + sx;
            if (t0 + t < T && sh.s_ok[t] != 0.0f)
                p.dbeta[((size_t)b * T + t0 + t) * p.Hv + hv] = sh.s_vec[2][t] + sh.s_vec[0][t];
        }
    } else if (tid == 0) {
        mbar_wait(&sh.bar2, mma_phase & 1u, nullptr);
    }
    if (tid == 0) bulk_wait_read();
    bc_teardown(tmem, 512);
}

// ===========================================================================
// launch 4: gradients II, one CTA per (chunk, hv, b): dQ^T, dK^T (M = Dk)
// ===========================================================================
constexpr uint32_t B_KQ = 0 * kSlot;    // K / Q (TMA)
constexpr uint32_t B_DY = 2 * kSlot;    // dY plain bf16 (TMA); then (dP o M)^T (bulk load)
constexpr uint32_t B_A = 3 * kSlot;     // S0^T, then G^T [128 dk][128 dv]; then K^T | Q^T [128 dk][64 i] x 2
constexpr uint32_t B_B = 7 * kSlot;     // [dY ; dZ] [128][128 dv]; then D [64 r][128 dv]
constexpr uint32_t B_B3 = 11 * kSlot;   // [dP o M ; H + H^T] (bulk load)
constexpr uint32_t kBSmem = 13 * kSlot + 1024;
// TMEM: S0^T [dY ; dZ]^T 0-127, (D G)^T 128-191, the (dP o M) and H products 256-383
constexpr uint32_t B_CQ1 = 0, B_CMG = 128, B_CR = 256;

__global__ void __launch_bounds__(kThreads, 1) bc_grad2_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                const __grid_constant__ CUtensorMap tm_q,
                                                                const __grid_constant__ CUtensorMap tm_dy,
                                                                const BcParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ BcShared sh;
    uint32_t base;
    uint8_t *sm = aligned_smem(smem_raw, base);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2, row = quad * 32 + lane;
    const int c = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
    const int hk = hv / (p.Hv / p.Hk);
    const int T = p.T, t0 = c * kC;
    if (!chunk_gates(p, sh, c, b, hv)) return;
    const uint32_t tmem = bc_setup(sh, 512);
    const uint32_t lt = tmem + ((uint32_t)(quad * 32) << 16);
    const size_t ci = chunk_index(p, b, hv, c);
    const uint8_t *out = p.img + ci * kImgBytes;

    if (tid == 0) {
        // k, q and dY tiles and B3: one arrival for the phase, with every byte
        mbar_expect_tx(&sh.bar0, kKQVBytes + 32768);
        issue_kq_tile(sm, B_KQ, B_DY, &tm_k, &tm_q, &tm_dy, p.Dk, p.Dv, hk, hv, b * T + t0, &sh.bar0);
        bulk_load(sm + B_B3, out + O_B3, 32768, &sh.bar0);
    }
    if (tid == 0) sh.s_scalar[0] = 0.0f;
    // S0^T and dZ into their tiles; G and D^T fetched now for the second
    // product; <G, S0> (the gamma_63 term of dlog g)
    float gv[64], dl[32];
    {
        float s0[64], z[32];
        load_rec128(p.rec_s + ci * kRec128, row, half, s0);
        load_rec64(p.rec_z + ci * kRec64, row, half, z);
        load_rec128(p.rec_g + ci * kRec128, row, half, gv);
        load_dt_record(p.rec_d + ci * kRec64, row, half, dl);
        put_transposed<64>(sm, B_A, 16384, 0, row, s0, half * 64);     // S0^T [dk][dv]
        put_transposed<32>(sm, B_B, 16384, 64, row, z, half * 32);     // dZ [r][dv], rows 64-127
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < 64; ++j) acc = fmaf(gv[j], s0[j], acc);
        acc = warp_sum(acc);
        __syncthreads();   // s_scalar zeroed
        if (lane == 0) atomicAdd(&sh.s_scalar[0], acc);
    }
    uint32_t mma_phase = 0;
    bool ok = wait_all(&sh.bar0, 0, p.err);
    bool dpmt_pending = false;
    if (ok) {
        build_dy_rows(sm, B_DY, B_B, 16384, sh.s_ok, tid);             // dY [r][dv], rows 0-63
        publish_operands();
        if (tid == 0) {
            // the dY slot is free: bring in (dP o M)^T
            mbar_expect_tx(&sh.bar1, 16384);
            bulk_load(sm + B_DY, out + O_DPMT, 16384, &sh.bar1);
            dpmt_pending = true;
            // [ (dY S0)^T | (dZ S0)^T ] = S0^T [dY ; dZ]^T
            const uint32_t id = umma::idesc(128, 128, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                umma::mma_tf32(tmem + B_CQ1, umma::desc_sw128(base + B_A + off), umma::desc_sw128(base + B_B + off), id,
                               k > 0);
            }
            umma::mma_commit(&sh.bar2);
        }
        ok = wait_all(&sh.bar2, mma_phase++ & 1u, p.err);
    }
    if (ok) {
        put_transposed<64>(sm, B_A, 16384, 0, row, gv, half * 64);     // G^T [dk][dv]
        put_transposed<32>(sm, B_B, 8192, 0, row, dl, half * 32);      // D [r][dv]
        publish_operands();
        if (tid == 0) {
            // (D G)^T = G^T D^T
            const uint32_t id = umma::idesc(128, 64, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                umma::mma_tf32(tmem + B_CMG, umma::desc_sw128(base + B_A + (k >> 2) * 16384 + (k & 3) * 32),
                               umma::desc_sw128(base + B_B + (k >> 2) * 8192 + (k & 3) * 32), id, k > 0);
            umma::mma_commit(&sh.bar2);
        }
        ok = wait_all(&sh.bar2, mma_phase++ & 1u, p.err);
    }
    if (ok) {
        build_xt(sm, B_KQ, 0, B_A, nullptr, 1.0f, tid);          // K^T [dk][i]
        build_xt(sm, B_KQ, 64, B_A + 32768, nullptr, 1.0f, tid); // Q^T [dk][i]
        ok = wait_all(&sh.bar1, 0, p.err);
        if (tid == 0) dpmt_pending = false;
    }
    if (ok) {
        publish_operands();
        if (tid == 0) {
            // [ (dPM K)^T | ((H + H^T) K)^T ] = K^T B3^T ; ((dPM)^T Q)^T += Q^T dPM
            const uint32_t id128 = umma::idesc(128, 128, umma::kFmtTF32), id64 = umma::idesc(128, 64, umma::kFmtTF32);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t kt = k >> 2, ko = (k & 3) * 32;
                umma::mma_tf32(tmem + B_CR, umma::desc_sw128(base + B_A + kt * kSlot + ko),
                               umma::desc_sw128(base + B_B3 + kt * kSlot + ko), id128, k > 0);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t kt = k >> 2, ko = (k & 3) * 32;
                umma::mma_tf32(tmem + B_CR + 64, umma::desc_sw128(base + B_A + 32768 + kt * kSlot + ko),
                               umma::desc_sw128(base + B_DY + kt * 8192 + ko), id64, true);
            }
            umma::mma_commit(&sh.bar2);
        }
        ok = wait_all(&sh.bar2, mma_phase++ & 1u, p.err);
    }
    if (ok) {
        // dQ^T and dK^T columns of this thread (dk = row; steps r = 32 half + j)
        float q1[32], k1[32], mg[32], ra[32], rb[32], fg[32];
        umma::tmem_ld32(lt + B_CQ1 + half * 32, q1);
        umma::tmem_ld32(lt + B_CQ1 + 64 + half * 32, k1);
        umma::tmem_ld32(lt + B_CMG + half * 32, mg);
        umma::tmem_ld32(lt + B_CR + half * 32, ra);
        umma::tmem_ld32(lt + B_CR + 64 + half * 32, rb);
        umma::tmem_ld_wait();
        const size_t qk_row = (size_t)p.Hk * p.Dk;
        const bool col_ok = row < p.Dk;   // padded columns past the head are not written
        float *dq0 = p.dq + ((size_t)b * T + t0) * qk_row + (size_t)hk * p.Dk + (col_ok ? row : 0);
        float *dk0 = p.dk + ((size_t)b * T + t0) * qk_row + (size_t)hk * p.Dk + (col_ok ? row : 0);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int r = half * 32 + j;
            const float fmg = sh.s_kc[r] * mg[j];
            fg[j] = fmg * kq_elem(sm, B_KQ, r, row);
            if (col_ok && t0 + r < T && sh.s_ok[r] != 0.0f) {
                atomicAdd(dq0 + (size_t)r * qk_row, fmaf(sh.s_gam[r], q1[j], ra[j]));
                atomicAdd(dk0 + (size_t)r * qk_row, fmaf(-sh.s_bg[r], k1[j], fmg) + rb[j]);
            }
        }
        sh.s_red[0][quad][half * 32 + lane] = transpose_sum32(fg);
        __syncthreads();
        if (tid < kC) sh.s_vec[1][tid] = (sh.s_red[0][0][tid] + sh.s_red[0][1][tid]) +
                                         (sh.s_red[0][2][tid] + sh.s_red[0][3][tid]);
        __syncthreads();
        if (tid < kC) {
            const int t = tid;
            float pre = 0.0f;
            for (int r = 0; r < t; ++r) pre += sh.s_vec[1][r];
            const float dlog = reinterpret_cast<const float *>(out + O_PART)[t] + pre + sh.s_scalar[0] * sh.s_gam[kC - 1];
            if (t0 + t < T && sh.s_ok[t] != 0.0f) p.dg[((size_t)b * T + t0 + t) * p.Hv + hv] = dlog / sh.s_g[t];
        }
    } else if (tid == 0) {
        mbar_wait(&sh.bar2, mma_phase & 1u, nullptr);
        if (dpmt_pending) mbar_wait(&sh.bar1, 0, nullptr);
    }
    bc_teardown(tmem, 512);
}

struct BcLayout {
    int nchunks;
    size_t n, region, rec_floats, flag_bytes;
};

BcLayout bc_layout(const Sizes &s) {
    BcLayout l;
    l.nchunks = (s.T + kC - 1) / kC;
    l.n = (size_t)s.B * s.Hv * l.nchunks;
    // the chain images also hold the two-pass forward's blobs and ready
    // flags (145 KiB and 4 bytes per chunk, the flags rounded up to 256
    // bytes), so the size does not depend on the device's SM count
    l.region = l.n * kImgBytes;
    l.rec_floats = 2 * kRec128 + 2 * kRec64;
    l.flag_bytes = (l.n * sizeof(int) + 255) & ~(size_t)255;   // the overlapped form's ready flags
    return l;
}

}  // namespace

size_t backward_chunked_workspace(const Sizes &s) {
    const BcLayout l = bc_layout(s);
    return row_order_workspace(s) + l.region + l.n * l.rec_floats * sizeof(float) + l.flag_bytes;
}

cudaError_t launch_backward_chunked(const Sizes &s, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                    const float *g, const float *beta, const float *state_in, const uint8_t *mask,
                                    const uint16_t *dy, const float *dstate_out, float *dq, float *dk, float *dv,
                                    float *dg, float *dbeta, float *dstate_in, void *ws, unsigned *err,
                                    cudaStream_t st) {
    if (s.Dk > kD || s.Dv > kD) return cudaErrorNotSupported;
    const size_t nqk = (size_t)s.B * s.T * s.Hk * s.Dk, nv = (size_t)s.B * s.T * s.Hv * s.Dv;
    const size_t ng = (size_t)s.B * s.T * s.Hv;
    cudaError_t e = cudaMemsetAsync(dq, 0, nqk * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dk, 0, nqk * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, nv * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dg, 0, ng * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dbeta, 0, ng * sizeof(float), st);
    if (e != cudaSuccess) return e;
    const BcLayout l = bc_layout(s);
    const int *order = nullptr;
    if (mask != nullptr && s.B > 1) {
        e = launch_row_order(s, mask, ws, st);
        if (e != cudaSuccess) return e;
        order = static_cast<const int *>(ws);
    }
    uint8_t *w = static_cast<uint8_t *>(ws) + row_order_workspace(s);
    // the forward in record mode writes no y; its y tensor map is encoded on
    // dy (the same shape), which nothing writes
    uint16_t *y = const_cast<uint16_t *>(dy);
    uint8_t *region = w;
    w += l.region;
    float *rec_s = reinterpret_cast<float *>(w);
    float *rec_d = rec_s + l.n * kRec128;
    float *rec_g = rec_d + l.n * kRec64;
    float *rec_z = rec_g + l.n * kRec128;
    int *ready = reinterpret_cast<int *>(rec_z + l.n * kRec64);

    // the forward, keeping every chunk's start state and D^T
    if (prefill_two_pass_workspace(s) > l.region) return cudaErrorInvalidValue;
    if (prefill_two_pass_pays(s))
        e = launch_prefill_two_pass(s, q, k, v, g, beta, state_in, nullptr, mask, order, y, region, err, st, rec_s,
                                    rec_d);
    else
        e = launch_prefill_chunked(s, q, k, v, g, beta, state_in, nullptr, mask, order, y, nullptr, nullptr, 0.0f,
                                   err, st, rec_s, rec_d);
    if (e != cudaSuccess) return e;

    ChunkMaps mk, mv;   // k, q and dY (in the v slot); v
    if (!encode_chunk_maps(&mk, s, q, k, dy, nullptr, y) || !encode_chunk_maps(&mv, s, q, k, v, nullptr, y))
        return cudaErrorInvalidValue;
    static unsigned long long set1 = 0, set2 = 0, set3 = 0, set4 = 0, set5 = 0;   // one bit per device
    constexpr uint32_t kOverlapSmem = kLSmem > kRSmem ? kLSmem : kRSmem;
    e = set_max_smem(set1, bc_image_kernel, kLSmem);
    if (e == cudaSuccess) e = set_max_smem(set2, bc_chain_kernel, kRSmem);
    if (e == cudaSuccess) e = set_max_smem(set3, bc_grad1_kernel, kASmem);
    if (e == cudaSuccess) e = set_max_smem(set4, bc_grad2_kernel, kBSmem);
    if (e == cudaSuccess) e = set_max_smem(set5, bc_overlap_kernel, kOverlapSmem);
    if (e != cudaSuccess) return e;
    BcParams p{g, beta, mask, order, rec_s, rec_d, rec_g, rec_z, region, dstate_out,
               dq, dk, dv, dg, dbeta, dstate_in, err, s.B, s.T, s.Hk, s.Hv, s.Dk, s.Dv, l.nchunks};
    const dim3 chunks(l.nchunks, s.Hv, s.B);
    // chain images and the reverse chain: overlapped in one cooperative launch
    // when the heads leave most SMs to the image producers, else two launches
    const int n_heads = s.B * s.Hv;
    int per_sm = 0;
    if (4 * n_heads <= num_sms() &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bc_overlap_kernel, kThreads, kOverlapSmem) ==
            cudaSuccess &&
        per_sm >= 1) {
        e = cudaMemsetAsync(ready, 0, l.n * sizeof(int), st);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(num_sms() * per_sm);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kOverlapSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, bc_overlap_kernel, mk.k, mk.q, mk.v, p, n_heads, ready);
        if (e != cudaSuccess) return e;
    } else {
        bc_image_kernel<<<chunks, kThreads, kLSmem, st>>>(mk.k, mk.q, mk.v, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        bc_chain_kernel<<<dim3(s.Hv, s.B), kThreads, kRSmem, st>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    bc_grad1_kernel<<<chunks, kThreads, kASmem, st>>>(mk.k, mk.q, mv.v, mk.v, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bc_grad2_kernel<<<chunks, kThreads, kBSmem, st>>>(mk.k, mk.q, mk.v, p);
    return cudaGetLastError();
}

}  // namespace gdn
