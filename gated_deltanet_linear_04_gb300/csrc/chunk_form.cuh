// Building blocks of the chunked (WY / UT-transform) form of the gated delta
// rule on the 5th-generation tensor cores, shared by the single-pass kernel
// (prefill_chunk.cu) and the two-pass kernels (prefill_chunk2.cu).
//
// The recurrence of "mlex 0.1.2, src/models/gated_delta.rs" (GatedDeltaNet::
// forward, per-timestep loop) and of the gated_delta_step kernel of "mlx-bun
// 0.4.0 -> 1.0.0, package/src/model/qwen3-delta.ts", re-blocked exactly into
// chunks of 64 steps.  For a chunk with start state S0 ([Dv, Dk]) and base-2
// log-decay prefix sums lg_r = sum_{i<=r} log2 g_i:
//   A[r,i] = beta_r 2^(lg_r - lg_i) (k_r . k_i), i < r;   T = (I + A)^-1
//   U = T diag(beta) V,   W = T diag(beta 2^lg) K,   D = U - W S0^T
//   Y = diag(2^lg) Q S0^T + (M o Q K^T) D,   M[r,i] = 2^(lg_r - lg_i), i <= r
//   S = 2^lg_63 S0 + D^T diag(2^(lg_63 - lg)) K
// (a masked step enters with g = 1, beta = 0).  Every product is issued in
// transposed form so that the MMA row count is M = 128 (= Dv or Dk) and an
// accumulator row is one TMEM lane:
//   [K;Q] K^T        bf16 x bf16  -> QK columns (rows 0-63 K K^T, 64-127 Q K^T)
//   U^T = (bV)^T T^T tf32         -> D columns
//   W^T = (bgK)^T T^T tf32        -> W columns
//   S0 (-W)^T    tf32             -> W columns; D^T = U^T + that, added in f32
//   Y^T = S0 (gQ)^T  tf32         -> Y columns
//   Y^T += D^T P^T   tf32         -> Y columns
//   S  += D^T Kc^T   tf32         -> S columns (S pre-scaled by 2^lg_63)
// The state products read S straight from TMEM as their A operand (tf32 by
// truncation); every other f32 operand is rounded to tf32 (to nearest, ties
// away from zero: umma::to_tf32) when it is written to shared memory.
//
// Threads: 256 (8 warps).  Warp w reaches TMEM lanes [32 (w % 4), +32): its
// thread `row` = 32 (w % 4) + lane is one accumulator row; `half` = w / 4
// picks which 32-column half of a 64-column accumulator it handles.
//
// Shared-memory tiles (offsets relative to a 1024-byte aligned base):
//   KQ  bf16, K rows 0-63 / Q rows 64-127, two 128B-swizzled K-halves of 64
//   V   plain [64][128] bf16
//   GQ  (g Q) [64][128] tf32, 4 swizzled K-tiles of 8 KiB
//   KT  Kc^T [128][64] tf32, 2 swizzled K-tiles of 16 KiB (as BV, BK, DT)
//   NW  -W [64][128] tf32, 4 K-tiles of 8 KiB
//   P   [64][64] tf32, 2 K-tiles of 8 KiB
#pragma once

#include "common.cuh"
#include "internal.h"
#include "umma.cuh"

namespace gdn {
namespace chunkform {

constexpr int kThreads = 256;
constexpr int kC = 64;          // chunk length
constexpr int kD = 128;         // Dk = Dv
constexpr uint32_t kSlot = 16384;

// TMEM columns
constexpr uint32_t C_QK = 0, C_D = 64, C_W = 128, C_Y = 192, C_S = 256;

// Tensor maps of the chunked kernels (host side).  The kernels always work on
// 128-wide tiles.  At a head size of 128 the maps are plain row-major views:
// k and q [B*T][Hk*128] with a [64 steps][64 channels] box, 128-byte swizzled
// (a chunk's tile is two boxes, channels 0-63 and 64-127 of the head); v and
// z [B*T][Hv*128] with a [64][128] box; y [B][T][Hv*128] with a [1][64][128]
// box.  Below 128 the head is a dimension of its own: k and q [B*T][Hk][Dk]
// with a [64][1][64] box, v and z [B*T][Hv][Dv] with a [64][1][128] box, y
// [B][T][Hv][Dv] with a [1][64][1][128] box; the boxes run past the head's
// channels, the loads read zeros there and the y store writes only the first
// Dv channels, so the padded rows and columns of every product are exact
// zeros and the results are those of the true sizes.
struct ChunkMaps {
    CUtensorMap k, q, v, z, y;
};

inline bool encode_chunk_maps(ChunkMaps *m, const Sizes &s, const uint16_t *q, const uint16_t *k,
                              const uint16_t *v, const uint16_t *z, uint16_t *y) {
    const uint64_t rows = (uint64_t)s.B * (uint64_t)s.T;
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B, ns = CU_TENSOR_MAP_SWIZZLE_NONE;
    bool ok = true;
    if (s.Dk == kD) {
        const uint64_t dk[2] = {(uint64_t)s.Hk * kD, rows};
        const uint32_t bk[2] = {64, (uint32_t)kC};
        ok = encode_tmap(&m->k, k, bf, 2, 2, dk, bk, sw) && encode_tmap(&m->q, q, bf, 2, 2, dk, bk, sw);
    } else {
        const uint64_t dk[3] = {(uint64_t)s.Dk, (uint64_t)s.Hk, rows};
        const uint32_t bk[3] = {64, 1, (uint32_t)kC};
        ok = encode_tmap(&m->k, k, bf, 2, 3, dk, bk, sw) && encode_tmap(&m->q, q, bf, 2, 3, dk, bk, sw);
    }
    if (!ok) return false;
    auto vmap = [&](CUtensorMap *t, const uint16_t *ptr) {
        if (s.Dv == kD) {
            const uint64_t dv[2] = {(uint64_t)s.Hv * kD, rows};
            const uint32_t bv[2] = {(uint32_t)kD, (uint32_t)kC};
            return encode_tmap(t, ptr, bf, 2, 2, dv, bv, ns);
        }
        const uint64_t dv[3] = {(uint64_t)s.Dv, (uint64_t)s.Hv, rows};
        const uint32_t bv[3] = {(uint32_t)kD, 1, (uint32_t)kC};
        return encode_tmap(t, ptr, bf, 2, 3, dv, bv, ns);
    };
    if (!vmap(&m->v, v)) return false;
    if (s.Dv == kD) {
        const uint64_t dy[3] = {(uint64_t)s.Hv * kD, (uint64_t)s.T, (uint64_t)s.B};
        const uint32_t by[3] = {(uint32_t)kD, (uint32_t)kC, 1};
        ok = encode_tmap(&m->y, y, bf, 2, 3, dy, by, ns);
    } else {
        const uint64_t dy[4] = {(uint64_t)s.Dv, (uint64_t)s.Hv, (uint64_t)s.T, (uint64_t)s.B};
        const uint32_t by[4] = {(uint32_t)kD, 1, (uint32_t)kC, 1};
        ok = encode_tmap(&m->y, y, bf, 2, 4, dy, by, ns);
    }
    if (!ok) return false;
    m->z = m->v;   // unused without the gated norm
    return z == nullptr || vmap(&m->z, z);
}

// Chunk c's k, q (128B-swizzled K-halves) and v tiles of head (hk, hv) of the
// rows starting at flat row `rowg` = b * T + c * 64 into the KQ and V slots
// (the maps' forms above: Dk, Dv of 128 or below).
__device__ __forceinline__ void load_chunk_tiles(uint8_t *sm, uint32_t kq_off, uint32_t v_off, const CUtensorMap *tm_k,
                                                 const CUtensorMap *tm_q, const CUtensorMap *tm_v, int Dk, int Dv,
                                                 int hk, int hv, int rowg, uint64_t *bar) {
    mbar_expect_tx(bar, 4 * 8192 + 16384);
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
    if (Dv == kD) tma_load_2d(sm + v_off, tm_v, hv * kD, rowg, bar);
    else tma_load_3d(sm + v_off, tm_v, 0, hv, rowg, bar);
}

// The chunk's [64 steps][128] tile of y (or z, for loads) of head hv at step
// t0 of batch row b, in the map form of the head size.
__device__ __forceinline__ void store_chunk_y(const CUtensorMap *tm_y, int Dv, int hv, int t0, int b,
                                              const uint8_t *src) {
    if (Dv == kD) tma_store_3d(tm_y, hv * kD, t0, b, src);
    else tma_store_4d(tm_y, 0, hv, t0, b, src);
}

__device__ __forceinline__ void load_chunk_z(uint8_t *dst, const CUtensorMap *tm_z, int Dv, int hv, int rowg,
                                             uint64_t *bar) {
    if (Dv == kD) tma_load_2d(dst, tm_z, hv * kD, rowg, bar);
    else tma_load_3d(dst, tm_z, 0, hv, rowg, bar);
}

// The f32 state of head (b, hv) between global memory and the S columns of
// TMEM: thread `row` (= dv) moves columns [64 half, +64) of its row; rows at
// or past Dv and columns at or past Dk are zeros in TMEM and are not stored.
__device__ __forceinline__ void state_to_tmem(const float *state_in, uint32_t s_tmem, int b, int hv, int Hv, int Dk,
                                              int Dv, int row, int half) {
    const bool row_ok = row < Dv && state_in != nullptr;
    const size_t off = (((size_t)b * Hv + hv) * Dv + row) * Dk;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        float r[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const int col = half * 64 + cc * 32 + j;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row_ok && col < Dk) x = *reinterpret_cast<const float4 *>(state_in + off + col);
            r[j] = x.x; r[j + 1] = x.y; r[j + 2] = x.z; r[j + 3] = x.w;
        }
        umma::tmem_st32(s_tmem + half * 64 + cc * 32, r);
    }
    umma::tmem_st_wait();
}

__device__ __forceinline__ void state_from_tmem(float *state_out, uint32_t s_tmem, int b, int hv, int Hv, int Dk,
                                                int Dv, int row, int half) {
    if (state_out == nullptr) return;
    const size_t off = (((size_t)b * Hv + hv) * Dv + row) * Dk;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        float sv[32];
        umma::tmem_ld32(s_tmem + half * 64 + cc * 32, sv);
        umma::tmem_ld_wait();
        if (row < Dv) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const int col = half * 64 + cc * 32 + j;
                if (col < Dk)
                    *reinterpret_cast<float4 *>(state_out + off + col) =
                        make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
            }
        }
    }
}

// A / T working matrix, row-major; groups of 4 columns are XOR-permuted by the
// row (r % 8) so that row-per-thread float4 stores spread over all banks while
// each aligned group of 4 stays contiguous for float4 loads.
__device__ __forceinline__ int aidx(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

// 2^x of a non-positive log-decay difference with the hardware base-2
// exponential (ex2.approx: relative error ~2^-22, far below the tf32 rounding
// these factors go through; results below 2^-126 flush to zero, which is the
// limit the decay takes anyway).  The precise library exp2f path measured ~3x
// slower for the 64 x 64 ratio matrices built every chunk.
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

__device__ __forceinline__ void st_tf32x4(uint8_t *base, uint32_t off, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(base + off) =
        make_float4(umma::to_tf32(a), umma::to_tf32(b), umma::to_tf32(c), umma::to_tf32(d));
}

// ---------------------------------------------------------------------------
// per-step factors (warp 0): lg (base-2 prefix sums), gamma = 2^lg,
// kc = 2^(lg_63 - lg), beta, beta * gamma
// ---------------------------------------------------------------------------
__device__ __forceinline__ void step_factors(int lane, const float *g, const float *beta, float *s_lg,
                                             float *s_gam, float *s_kc, float *s_beta, float *s_bg) {
    const float la = log2_gate(g[2 * lane]), lb = log2_gate(g[2 * lane + 1]);
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
    const float b0 = beta[2 * lane], b1 = beta[2 * lane + 1];
    s_beta[2 * lane] = b0;
    s_beta[2 * lane + 1] = b1;
    s_bg[2 * lane] = b0 * e0;
    s_bg[2 * lane + 1] = b1 * e1;
}

// ---------------------------------------------------------------------------
// operand builds (all threads)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float kq_elem(const uint8_t *sm, uint32_t kq_off, int row, int dk) {
    // row 0-63: K, 64-127: Q; bf16, 128B swizzle, K-halves of 64 in two slots
    const uint16_t *p = reinterpret_cast<const uint16_t *>(
        sm + kq_off + (dk >> 6) * kSlot + umma::sw128((uint32_t)row, (uint32_t)(dk & 63) * 2));
    return bf16_to_f32(*p);
}

// (g Q)[r][dk]: a warp covers one row r, 4 consecutive dk per lane
__device__ __forceinline__ void build_gq(uint8_t *sm, uint32_t kq_off, uint32_t gq_off, const float *s_gam,
                                         int tid) {
    for (int i = tid; i < kC * kD / 4; i += kThreads) {
        const int r = i >> 5, dk = (i & 31) * 4;
        const float gm = s_gam[r];
        const uint2 qq = *reinterpret_cast<const uint2 *>(
            sm + kq_off + (dk >> 6) * kSlot + umma::sw128(64 + r, (dk & 63) * 2));
        st_tf32x4(sm, gq_off + (dk >> 5) * 8192 + umma::sw128(r, (dk & 31) * 4), gm * __uint_as_float(qq.x << 16),
                  gm * __uint_as_float(qq.x & 0xffff0000u), gm * __uint_as_float(qq.y << 16),
                  gm * __uint_as_float(qq.y & 0xffff0000u));
    }
}

// Kc^T[dk][r] and (b g K)^T[dk][r]: lanes take consecutive dk (conflict-free
// reads along a K row and conflict-free 16-byte stores, a quarter-warp's
// eight dk rows on eight swizzle phases), each thread 4 consecutive r of two
// row quads (warp w: rows 4w and 4w + 32), so the per-row factors are loaded
// once per quad rather than once per element group
__device__ __forceinline__ void build_kt_bk(uint8_t *sm, uint32_t kq_off, uint32_t kt_off, uint32_t bk_off,
                                            const float *s_kc, const float *s_bg, int tid) {
    const int lane = tid & 31, w = tid >> 5;
#pragma unroll
    for (int rp = 0; rp < 2; ++rp) {
        const int r = (w + 8 * rp) * 4;
        const float4 kc = ld4(s_kc + r), bg = ld4(s_bg + r);
#pragma unroll
        for (int j = 0; j < kD / 32; ++j) {
            const int dk = lane + 32 * j;
            const float k0 = kq_elem(sm, kq_off, r, dk), k1 = kq_elem(sm, kq_off, r + 1, dk),
                        k2 = kq_elem(sm, kq_off, r + 2, dk), k3 = kq_elem(sm, kq_off, r + 3, dk);
            const uint32_t off = (r >> 5) * kSlot + umma::sw128(dk, (r & 31) * 4);
            st_tf32x4(sm, kt_off + off, kc.x * k0, kc.y * k1, kc.z * k2, kc.w * k3);
            st_tf32x4(sm, bk_off + off, bg.x * k0, bg.y * k1, bg.z * k2, bg.w * k3);
        }
    }
}

// (b V)^T[dv][i]: the same thread layout
__device__ __forceinline__ void build_bv(uint8_t *sm, uint32_t v_off, uint32_t bv_off, const float *s_beta,
                                         int tid) {
    const uint16_t *Vs = reinterpret_cast<const uint16_t *>(sm + v_off);
    const int lane = tid & 31, w = tid >> 5;
#pragma unroll
    for (int rp = 0; rp < 2; ++rp) {
        const int r = (w + 8 * rp) * 4;
        const float4 be = ld4(s_beta + r);
#pragma unroll
        for (int j = 0; j < kD / 32; ++j) {
            const int dv = lane + 32 * j;
            st_tf32x4(sm, bv_off + (r >> 5) * kSlot + umma::sw128(dv, (r & 31) * 4),
                      be.x * bf16_to_f32(Vs[r * kD + dv]), be.y * bf16_to_f32(Vs[(r + 1) * kD + dv]),
                      be.z * bf16_to_f32(Vs[(r + 2) * kD + dv]), be.w * bf16_to_f32(Vs[(r + 3) * kD + dv]));
        }
    }
}

// A from the K K^T rows (0-63) of the QK accumulator; threads of TMEM quads 0-1
__device__ __forceinline__ void build_a(uint32_t qk_tmem, float *As, const float *s_lg, const float *s_beta,
                                        int row, int half) {
    float kk[32];
    umma::tmem_ld32(qk_tmem + half * 32, kk);
    umma::tmem_ld_wait();
    const int r = row;   // 0..63
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

// P = M o Q K^T from the Q K^T row (64-127) of the QK accumulator held in
// registers (threads of TMEM quads 2-3)
__device__ __forceinline__ void p_tile(const float (&qk)[32], uint8_t *sm, uint32_t p_off, const float *s_lg,
                                       int row, int half) {
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
        st_tf32x4(sm, p_off + half * 8192 + umma::sw128(r, j * 4), v4[0], v4[1], v4[2], v4[3]);
    }
}

// ---------------------------------------------------------------------------
// T = (I + A)^-1 in place, by blocked doubling (all threads; block barriers)
// ---------------------------------------------------------------------------

// One merge level: for each pair of S x S diagonal blocks (a = [q0, q0+S),
// b = [q0+S, q0+2S)) of the unit lower triangular T, the lower-left block is
// X = -T_bb A_ba T_aa.  Sums run over full blocks because the triangular
// factors hold explicit zeros above the diagonal.  A work item computes 4
// adjacent columns of RB rows, rows rg, rg + S/RB, ..., so that each loaded
// row of the right factor serves RB rows, and the rows a warp reads the left
// factor from at once differ in (row mod 8), i.e. in their bank swizzle.
// Each output element is the same sequence of fused multiply-adds as with
// one row per thread.  At S = 32 (cycles per level in an instrumented copy):
// one row per thread (256 threads, every warp loading the whole right
// factor) 2.8k, four rows (64 threads, too few to hide the load latency)
// 2.5k, two rows (128 threads) 1.9k.
template <int S, int RB>
__device__ __forceinline__ void merge_level(float *As, float *Ys, int tid) {
    constexpr int G4 = S / 4;          // column groups of 4
    constexpr int RG = S / RB;         // row groups
    constexpr int NT = (32 / S) * RG * G4;
    const int pi = tid / (RG * G4), rem = tid % (RG * G4), rg = rem / G4, c = (rem % G4) * 4, q0 = pi * 2 * S;
    if (tid < NT) {
        // packed two-wide FMAs: each half rounds like fmaf
        float2 lo[RB], hi[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) lo[i] = hi[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < S; ++m) {
            const float4 t = ld4(As + aidx(q0 + m, q0 + c));
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const float a = As[aidx(q0 + S + rg + i * RG, q0 + m)];
                lo[i] = __ffma2_rn(make_float2(a, a), make_float2(t.x, t.y), lo[i]);
                hi[i] = __ffma2_rn(make_float2(a, a), make_float2(t.z, t.w), hi[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < RB; ++i)
            st4(Ys + (pi * S + rg + i * RG) * S + c, make_float4(lo[i].x, lo[i].y, hi[i].x, hi[i].y));
    }
    __syncthreads();
    if (tid < NT) {
        float2 lo[RB], hi[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) lo[i] = hi[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < S; ++m) {
            const float4 yv = ld4(Ys + (pi * S + m) * S + c);
#pragma unroll
            for (int i = 0; i < RB; ++i) {
                const float t = As[aidx(q0 + S + rg + i * RG, q0 + S + m)];
                lo[i] = __ffma2_rn(make_float2(t, t), make_float2(yv.x, yv.y), lo[i]);
                hi[i] = __ffma2_rn(make_float2(t, t), make_float2(yv.z, yv.w), hi[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < RB; ++i)
            st4(As + aidx(q0 + S + rg + i * RG, q0 + c), make_float4(-lo[i].x, -lo[i].y, -hi[i].x, -hi[i].y));
    }
    __syncthreads();
}

__device__ __forceinline__ void invert_unit_lower(float *As, float *Ys, int tid) {
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
    merge_level<8, 1>(As, Ys, tid);
    merge_level<16, 2>(As, Ys, tid);
    merge_level<32, 2>(As, Ys, tid);
}

// T -> tf32 B operand [r][i] (2 K-tiles of 8 KiB)
__device__ __forceinline__ void t_to_tf32(const float *As, uint8_t *sm, uint32_t t_off, int tid) {
    for (int i = tid; i < kC * kC / 4; i += kThreads) {
        const int r = i >> 4, c4 = (i & 15) * 4;
        const float4 tv = ld4(As + aidx(r, c4));
        st_tf32x4(sm, t_off + (c4 >> 5) * 8192 + umma::sw128(r, (c4 & 31) * 4), tv.x, tv.y, tv.z, tv.w);
    }
}

// -W (tf32) from the W accumulator: thread `row` is dk, its half covers 32 r
__device__ __forceinline__ void neg_w_tile(uint32_t w_tmem, uint8_t *sm, uint32_t nw_off, int row, int half) {
    float wv[32];
    umma::tmem_ld32(w_tmem + half * 32, wv);
    umma::tmem_ld_wait();
    const int dk = row;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int r = half * 32 + j;
        *reinterpret_cast<float *>(sm + nw_off + (dk >> 5) * 8192 + umma::sw128(r, (dk & 31) * 4)) =
            umma::to_tf32(-wv[j]);
    }
}

// D^T (tf32 A operand) from a D accumulator row held in registers
__device__ __forceinline__ void dt_tile(const float (&dv)[32], uint8_t *sm, uint32_t dt_off, int row, int half) {
#pragma unroll
    for (int j = 0; j < 32; j += 4)
        st_tf32x4(sm, dt_off + half * kSlot + umma::sw128(row, j * 4), dv[j], dv[j + 1], dv[j + 2], dv[j + 3]);
}

// ---------------------------------------------------------------------------
// per-chunk records for the chunked backward (global memory, f32), in the
// order the 256 threads of a chunk CTA hold them: thread (row, half) keeps
// the 64 columns [64 half, +64) of TMEM lane `row` of a [128][128] matrix
// (float4 j of them at float4 index (16 half + j) 128 + row), or the 32
// columns [32 half, +32) of a [128][64] one (float4 index (8 half + j) 128 +
// row), so that a warp touches 512 contiguous bytes per access.
// ---------------------------------------------------------------------------
constexpr size_t kRec128 = 128 * 128, kRec64 = 128 * 64;   // floats per record

__device__ __forceinline__ float4 *rec128_at(float *rec, int row, int half, int j) {
    return reinterpret_cast<float4 *>(rec) + ((half * 16 + j) * 128 + row);
}
__device__ __forceinline__ const float4 *rec128_at(const float *rec, int row, int half, int j) {
    return reinterpret_cast<const float4 *>(rec) + ((half * 16 + j) * 128 + row);
}
__device__ __forceinline__ float4 *rec64_at(float *rec, int row, int half, int j) {
    return reinterpret_cast<float4 *>(rec) + ((half * 8 + j) * 128 + row);
}
__device__ __forceinline__ const float4 *rec64_at(const float *rec, int row, int half, int j) {
    return reinterpret_cast<const float4 *>(rec) + ((half * 8 + j) * 128 + row);
}

// The D^T record is the shared-memory D^T operand tile itself (dt_tile
// below: [128 dv][64 r] tf32, two 128B-swizzled K-tiles of 16 KiB), bulk-
// stored as it is; thread (row, half) reads its 32 columns [32 half, +32)
// back from row `row` of K-tile `half` (16-byte group j at j ^ (row % 8)).
__device__ __forceinline__ void load_dt_record(const float *rec, int row, int half, float (&v)[32]) {
    const float4 *base = reinterpret_cast<const float4 *>(rec) + half * 1024 + row * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 x = base[j ^ (row & 7)];
        v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
    }
}

// a [128][64] record row held in registers (32 columns of this thread)
__device__ __forceinline__ void store_rec64(float *rec, int row, int half, const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        *rec64_at(rec, row, half, j) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

// S <- gl S in TMEM (the products that read S0 must have completed); both
// halves of the thread's 64 columns are loaded before one wait.  With `rec`,
// S before the decay (the chunk's start state) is also stored as a record.
__device__ __forceinline__ void decay_state(uint32_t s_tmem, float gl, int half, float *rec = nullptr,
                                            int row = 0) {
    float sa[32], sb[32];
    umma::tmem_ld32(s_tmem + half * 64, sa);
    umma::tmem_ld32(s_tmem + half * 64 + 32, sb);
    umma::tmem_ld_wait();
    if (rec != nullptr) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            *rec128_at(rec, row, half, j) = make_float4(sa[4 * j], sa[4 * j + 1], sa[4 * j + 2], sa[4 * j + 3]);
            *rec128_at(rec, row, half, 8 + j) = make_float4(sb[4 * j], sb[4 * j + 1], sb[4 * j + 2], sb[4 * j + 3]);
        }
    }
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float2 a2 = __fmul2_rn(make_float2(sa[j], sa[j + 1]), make_float2(gl, gl));
        const float2 b2 = __fmul2_rn(make_float2(sb[j], sb[j + 1]), make_float2(gl, gl));
        sa[j] = a2.x; sa[j + 1] = a2.y;
        sb[j] = b2.x; sb[j + 1] = b2.y;
    }
    umma::tmem_st32(s_tmem + half * 64, sa);
    umma::tmem_st32(s_tmem + half * 64 + 32, sb);
}

// ---------------------------------------------------------------------------
// tensor-core issue (one thread; the caller commits)
// ---------------------------------------------------------------------------
// [K;Q] K^T (bf16, M = 128, N = 64, K = 128)
__device__ __forceinline__ void issue_kq(uint32_t tmem, uint32_t base, uint32_t kq_off) {
    const uint32_t id = umma::idesc(128, 64, umma::kFmtBF16);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t a = base + kq_off + (k >> 2) * kSlot + (k & 3) * 32;
        umma::mma_bf16(tmem + C_QK, umma::desc_sw128(a), umma::desc_sw128(a), id, k > 0);
    }
}

// U^T = (bV)^T T^T and W^T = (bgK)^T T^T (tf32, M = 128, N = 64, K = 64)
__device__ __forceinline__ void issue_uw(uint32_t tmem, uint32_t base, uint32_t t_off, uint32_t bv_off,
                                         uint32_t bk_off) {
    const uint32_t id = umma::idesc(128, 64, umma::kFmtTF32);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t kt = k >> 2, ko = (k & 3) * 32;
        const uint64_t bt = umma::desc_sw128(base + t_off + kt * 8192 + ko);
        umma::mma_tf32(tmem + C_D, umma::desc_sw128(base + bv_off + kt * kSlot + ko), bt, id, k > 0);
        umma::mma_tf32(tmem + C_W, umma::desc_sw128(base + bk_off + kt * kSlot + ko), bt, id, k > 0);
    }
}

// S0 (-W)^T into the W columns (free once -W has been read out) and
// Y^T = S0 (gQ)^T, S0 read from TMEM (tf32, K = 128); D^T = U^T + S0 (-W)^T
// is then formed in f32 by the threads that build the D^T tile
__device__ __forceinline__ void issue_s0_products(uint32_t tmem, uint32_t base, uint32_t nw_off,
                                                  uint32_t gq_off) {
    const uint32_t id = umma::idesc(128, 64, umma::kFmtTF32);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint32_t kt = k >> 2, ko = (k & 3) * 32, a = tmem + C_S + 8 * k;
        umma::mma_tf32_tmem_a(tmem + C_W, a, umma::desc_sw128(base + nw_off + kt * 8192 + ko), id, k > 0);
        umma::mma_tf32_tmem_a(tmem + C_Y, a, umma::desc_sw128(base + gq_off + kt * 8192 + ko), id, k > 0);
    }
}

// Y^T += D^T P^T and S += D^T Kc^T (tf32, K = 64)
__device__ __forceinline__ void issue_dt_products(uint32_t tmem, uint32_t base, uint32_t dt_off, uint32_t p_off,
                                                  uint32_t kt_off) {
    const uint32_t idy = umma::idesc(128, 64, umma::kFmtTF32);
    const uint32_t ids = umma::idesc(128, 128, umma::kFmtTF32);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t kt = k >> 2, ko = (k & 3) * 32;
        const uint64_t a = umma::desc_sw128(base + dt_off + kt * kSlot + ko);
        umma::mma_tf32(tmem + C_Y, a, umma::desc_sw128(base + p_off + kt * 8192 + ko), idy, true);
        umma::mma_tf32(tmem + C_S, a, umma::desc_sw128(base + kt_off + kt * kSlot + ko), ids, true);
    }
}

// y of the chunk from the Y accumulator into a bf16 staging tile [64 steps][128 dv]
// (masked steps are written as zeros).  Thread `row` holds one dv for 32
// steps; the lanes of a pair (dv even, dv + 1) swap one value per two steps,
// so that each writes two adjacent dv of one step as one 32-bit word.
__device__ __forceinline__ void stage_y(uint32_t y_tmem, uint8_t *sm, uint32_t yst_off, const int *s_m, int row,
                                        int half) {
    float yv[32];
    umma::tmem_ld32(y_tmem + half * 32, yv);
    const unsigned valid = __ballot_sync(0xffffffffu, s_m[half * 32 + (threadIdx.x & 31)] != 0);
    umma::tmem_ld_wait();
    uint32_t *Yst = reinterpret_cast<uint32_t *>(sm + yst_off);
    const bool odd = (row & 1) != 0;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        // even lanes keep step j and receive the partner's; odd lanes step j + 1
        const float mine = odd ? yv[j + 1] : yv[j];
        const float other = __shfl_xor_sync(0xffffffffu, odd ? yv[j] : yv[j + 1], 1);
        const int r = half * 32 + j + (odd ? 1 : 0);
        const bool m = (valid >> (j + (odd ? 1 : 0))) & 1u;
        const float lo = odd ? other : mine, hi = odd ? mine : other;
        const __nv_bfloat162 h = __floats2bfloat162_rn(m ? lo : 0.0f, m ? hi : 0.0f);
        Yst[(r * kD + (row & ~1)) >> 1] = *reinterpret_cast<const uint32_t *>(&h);
    }
}

}  // namespace chunkform
}  // namespace gdn
