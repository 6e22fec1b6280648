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
// The rows of S (and of dS) evolve independently, and the dS recursion
// (dS += dy q^T, du = beta dS k, dS = g (dS - du k^T)) needs neither S nor v.
// So the work splits into two launches:
//  1. sweeps, one CTA (4 warps) per 32 state rows of a head and direction:
//     the forward sweep stores S at the start of every 32-step chunk, the
//     reverse sweep stores dS at the end of every chunk (and dS of the
//     initial state, the output dstate_in); the two run side by side, each
//     loading the next chunk's inputs into registers while it steps through
//     the current one.
//  2. chunks, every (row slice, head, chunk) independently on a fixed grid
//     of CTAs that each own a 32-step history buffer: from the chunk's S it
//     recomputes the chunk's states into the history buffer (global memory,
//     read back while it is still in L2 as far as it fits), keeping u per
//     row in shared memory, then runs the full reverse steps from the
//     chunk's end dS with dS in registers.
// Every CTA walks only the chunks from its row's first to its last valid
// step, and with a mask the rows are handed out longest first.
// Lane (rg, cg) of warp w holds rows w*8 + rg*2 + {0, 1} and the Dk/8
// columns of the 16-byte column groups cg, cg + 8, ... (see Lanes), so a
// row's dot product is a 3-level shuffle sum over the 8 lanes sharing rg.  The sums over rows (dq, dk, dg, dbeta) are
// reduced within the warp, collected per step in shared memory and added to
// the outputs with atomics once per chunk; the atomics also sum over the
// row slices and over the v-heads that share a k-head.  The call zeroes the
// outputs first.  Where the row slices alone fill the GPU (two or more per
// SM) the split buys no parallelism and costs the second sweep, so one
// launch runs, per slice, the forward sweep and then the chunks in reverse,
// carrying dS from chunk to chunk.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 128;
constexpr int kRows = 32;        // state rows per CTA
constexpr int kC = 32;           // steps per staged chunk (checkpoint interval, history length)

struct BwdParams {
    const uint16_t *q, *k, *v;
    const float *g, *beta, *state_in;
    const uint8_t *mask;
    const uint16_t *dy;
    const float *dstate_out;
    float *dq, *dk, *dv, *dg, *dbeta, *dstate_in;
    float *ck;      // S at the start of every chunk   [B, Hv, slices, nck, kRows, Dk]
    float *dck;     // dS at the end of every chunk    [B, Hv, slices, nck, kRows, Dk] (split form)
    float *hist;    // one [kC, kRows, Dk] history per chunk-pass CTA
    const int *order;   // row slot -> batch row, longest first (masked batches), or null
    int B, T, Hk, Hv, Dv, nck;
};

template <int DK>
struct BwdSmem {
    float q[kC][DK], k[kC][DK];
    float v[kC][kRows], dy[kC][kRows], u[kC][kRows];
    float g[kC], beta[kC];
    int m[kC];
    // per-step column sums of dq (at red_q(col)) and dk (at red_k(col)); see
    // red_q / red_k below for the layout
    float red[kC][2 * DK + 8];
    float red_g[kC], red_b[kC];
    int range[2];   // first and last valid step of the row (valid_chunks)
};

// Index of column c's dq / dk sum in a row of BwdSmem::red.  After the
// transpose-reduction the four row groups of a warp add, for the same column
// lane, dq of the lower column half (rg 0), dk of the lower half (rg 1), dq of
// the upper half (rg 2) and dk of the upper half (rg 3): the k half starts one
// bank over and (for Dk >= 64) the upper half is skewed by two banks, so the
// four land on different banks.
template <int DK>
__device__ __forceinline__ int red_q(int c) { return DK >= 64 ? c + ((c >= DK / 2) ? 2 : 0) : c; }
template <int DK>
__device__ __forceinline__ int red_k(int c) { return DK + 5 + red_q<DK>(c); }

// One chunk's inputs on their way from global to shared memory: each
// thread's share of the q / k rows (4 columns per word) and of the v / dy
// entries of the CTA's rows, and (threads < kC) one step's g, beta, mask.
template <int DK>
struct ChunkRegs {
    static constexpr int NQK = kC * DK / 4 / kThreads;
    static constexpr int NV = kC * kRows / kThreads;
    static_assert(NQK * 4 * kThreads == kC * DK && NV * kThreads == kC * kRows, "chunk does not split evenly");
    uint2 k[NQK], q[NQK];
    uint16_t v[NV], dy[NV];
    float g, beta;
    int m;
};

// Loads steps [t0, t0 + kC) of the chunk: q, k of the k-head, v and dy of the
// CTA's rows, g, beta, the mask (steps past T or masked: m = 0; past T the
// values are zeros, g one).  with_q_dy = false for the forward direction
// (q and dy left zero).  No shared memory is touched, so the loads of the
// next chunk can be in flight while the current one is stepped through.
template <int DK>
__device__ __forceinline__ void fetch_chunk(const BwdParams &p, ChunkRegs<DK> &r, int b, int hk, int hv, int r0,
                                            int t0, bool with_q_dy) {
    const int tid = threadIdx.x;
    const int T = p.T;
    constexpr int V4 = DK / 4;
#pragma unroll
    for (int n = 0; n < ChunkRegs<DK>::NQK; ++n) {
        const int i = tid + n * kThreads;
        const int t = t0 + i / V4, c4 = (i % V4) * 4;
        r.k[n] = r.q[n] = make_uint2(0u, 0u);
        if (t < T) {
            const size_t off = (((size_t)b * T + t) * p.Hk + hk) * DK + c4;
            r.k[n] = *reinterpret_cast<const uint2 *>(p.k + off);
            if (with_q_dy) r.q[n] = *reinterpret_cast<const uint2 *>(p.q + off);
        }
    }
#pragma unroll
    for (int n = 0; n < ChunkRegs<DK>::NV; ++n) {
        const int i = tid + n * kThreads;
        const int t = t0 + i / kRows, rr = i % kRows;
        r.v[n] = r.dy[n] = 0;
        if (t < T) {
            const size_t off = (((size_t)b * T + t) * p.Hv + hv) * p.Dv + r0 + rr;
            r.v[n] = p.v[off];
            if (with_q_dy) r.dy[n] = p.dy[off];
        }
    }
    r.m = 0;
    r.g = 1.0f;
    r.beta = 0.0f;
    if (tid < kC && t0 + tid < T) {
        const int t = t0 + tid;
        r.m = p.mask == nullptr ? 1 : (p.mask[(size_t)b * T + t] != 0);
        const size_t gi = ((size_t)b * T + t) * p.Hv + hv;
        r.g = p.g[gi];
        r.beta = p.beta[gi];
    }
}

// Writes a fetched chunk to shared memory as f32 (q / k rows with 16-byte
// stores).  The caller synchronises before and after.
template <int DK>
__device__ __forceinline__ void commit_chunk(BwdSmem<DK> &s, const ChunkRegs<DK> &r) {
    const int tid = threadIdx.x;
    constexpr int V4 = DK / 4;
#pragma unroll
    for (int n = 0; n < ChunkRegs<DK>::NQK; ++n) {
        const int i = tid + n * kThreads;
        const int tl = i / V4, c4 = (i % V4) * 4;
        const uint2 kk = r.k[n], qq = r.q[n];
        *reinterpret_cast<float4 *>(&s.k[tl][c4]) =
            make_float4(__uint_as_float(kk.x << 16), __uint_as_float(kk.x & 0xffff0000u),
                        __uint_as_float(kk.y << 16), __uint_as_float(kk.y & 0xffff0000u));
        *reinterpret_cast<float4 *>(&s.q[tl][c4]) =
            make_float4(__uint_as_float(qq.x << 16), __uint_as_float(qq.x & 0xffff0000u),
                        __uint_as_float(qq.y << 16), __uint_as_float(qq.y & 0xffff0000u));
    }
#pragma unroll
    for (int n = 0; n < ChunkRegs<DK>::NV; ++n) {
        const int i = tid + n * kThreads;
        s.v[i / kRows][i % kRows] = bf16_to_f32(r.v[n]);
        s.dy[i / kRows][i % kRows] = bf16_to_f32(r.dy[n]);
    }
    if (tid < kC) {
        s.m[tid] = r.m;
        s.g[tid] = r.g;
        s.beta[tid] = r.beta;
    }
}

// Stages the chunk at t0 (fetch, then commit).  Block-wide; ends with a
// barrier.
template <int DK>
__device__ __forceinline__ void stage_chunk(const BwdParams &p, BwdSmem<DK> &s, int b, int hk, int hv, int r0,
                                            int t0, bool with_q_dy) {
    ChunkRegs<DK> r;
    fetch_chunk<DK>(p, r, b, hk, hv, r0, t0, with_q_dy);
    commit_chunk<DK>(s, r);
    __syncthreads();
}

// Whether steps [t0, t0 + kC) of row b hold a valid step (uniform over the CTA).
__device__ __forceinline__ bool chunk_active(const BwdParams &p, int b, int t0) {
    if (p.mask == nullptr) return true;
    const int t = t0 + (int)threadIdx.x;
    const bool m = threadIdx.x < kC && t < p.T && p.mask[(size_t)b * p.T + t] != 0;
    return __syncthreads_or(m) != 0;
}

// The chunks [c_begin, c_end) of row b from its first to its last valid
// step ([0, nck) without a mask; empty for a wholly masked row): outside them
// the state and its gradient pass through unchanged.  Block-wide.
template <int DK>
__device__ __forceinline__ void valid_chunks(const BwdParams &p, BwdSmem<DK> &s, int b, int &c_begin, int &c_end) {
    if (p.mask == nullptr) {
        c_begin = 0;
        c_end = p.nck;
        return;
    }
    if (threadIdx.x == 0) {
        s.range[0] = INT_MAX;
        s.range[1] = -1;
    }
    __syncthreads();
    const uint8_t *mrow = p.mask + (size_t)b * p.T;
    int lo = INT_MAX, hi = -1;
#pragma unroll 8
    for (int t = threadIdx.x; t < p.T; t += kThreads)
        if (mrow[t] != 0) {
            lo = min(lo, t);
            hi = t;
        }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if ((threadIdx.x & 31u) == 0) {
        atomicMin(&s.range[0], lo);
        atomicMax(&s.range[1], hi);
    }
    __syncthreads();
    lo = s.range[0];
    hi = s.range[1];
    __syncthreads();
    c_begin = hi < 0 ? 0 : lo / kC;
    c_end = hi < 0 ? 0 : hi / kC + 1;
}

// Four partial sums of a dot product (the lane's columns j with j % 4 = 0..3,
// four independent chains instead of one) added in a fixed order.
__device__ __forceinline__ float sum4(const float (&x)[4]) { return (x[0] + x[1]) + (x[2] + x[3]); }

// sum over the 8 lanes of a row group (lanes differing in bits 0-2)
__device__ __forceinline__ float row_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
}

// The two rows and Dk/8 columns of the state that one lane holds: rows
// rl[0], rl[1] of the CTA's slice and the 16-byte column groups cg, cg + 8,
// ... (element j at column col(j)), so the eight column lanes of a row read a
// staged q / k row as 8 consecutive 16-byte words, free of bank conflicts.
template <int DK>
struct Lanes {
    static constexpr int CW = DK / 8;
    int lane, rg, cg, rl[2];

    __device__ __forceinline__ Lanes() {
        lane = threadIdx.x & 31;
        rg = lane >> 3;
        cg = lane & 7;
        rl[0] = (int)(threadIdx.x >> 5) * 8 + rg * 2;
        rl[1] = rl[0] + 1;
    }
    __device__ __forceinline__ int col(int j) const { return ((cg + 8 * (j >> 2)) << 2) + (j & 3); }
    __device__ __forceinline__ void load(const float *src, float (&x)[2][CW]) const {   // src: [kRows][DK]
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < CW; j += 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(src + (size_t)rl[i] * DK + col(j));
                x[i][j] = v4.x; x[i][j + 1] = v4.y; x[i][j + 2] = v4.z; x[i][j + 3] = v4.w;
            }
    }
    __device__ __forceinline__ void store(float *dst, const float (&x)[2][CW]) const {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < CW; j += 4)
                *reinterpret_cast<float4 *>(dst + (size_t)rl[i] * DK + col(j)) =
                    make_float4(x[i][j], x[i][j + 1], x[i][j + 2], x[i][j + 3]);
    }
    // the slice of a [Dv, DK] head array (or zeros for a null one)
    __device__ __forceinline__ void load_or_zero(const float *src, float (&x)[2][CW]) const {
        if (src != nullptr) {
            load(src, x);
            return;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < CW; ++j) x[i][j] = 0.0f;
    }
};

// One forward step of the lane's two rows from the staged chunk; returns u
// per row.
// The step loops below run on adjacent column pairs (j, j + 1 with j even:
// the lane's columns come in runs of four) with the packed two-wide f32
// instructions; each half rounds like the scalar instruction and the four
// partial sums keep their order, so every value is the scalar loop's.
__device__ __forceinline__ float2 pair(const float *x, int j) { return make_float2(x[j], x[j + 1]); }

template <int DK>
__device__ __forceinline__ void fwd_step(const BwdSmem<DK> &s, const Lanes<DK> &L, float (&S)[2][DK / 8], int tl,
                                         float (&u)[2]) {
    constexpr int CW = DK / 8;
    const float gg = s.g[tl], bb = s.beta[tl];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float2 kv01 = make_float2(0.0f, 0.0f), kv23 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < CW; j += 4) {
            kv01 = __ffma2_rn(pair(S[i], j), pair(s.k[tl], L.col(j)), kv01);
            kv23 = __ffma2_rn(pair(S[i], j + 2), pair(s.k[tl], L.col(j + 2)), kv23);
        }
        const float kv4[4] = {kv01.x, kv01.y, kv23.x, kv23.y};
        const float kv = gg * row_sum(sum4(kv4));
        u[i] = s.v[tl][L.rl[i]] - kv;
        const float dl = bb * u[i];
        const float2 g2 = make_float2(gg, gg), dl2 = make_float2(dl, dl);
#pragma unroll
        for (int j = 0; j < CW; j += 2) {
            const float2 r = __ffma2_rn(dl2, pair(s.k[tl], L.col(j)), __fmul2_rn(g2, pair(S[i], j)));
            S[i][j] = r.x;
            S[i][j + 1] = r.y;
        }
    }
}

// One reverse step of dS alone: dS += dy q^T, ddelta = dS k, du = beta
// ddelta, dS = g (dS - du k^T), in the operation order of the full reverse
// step below, so both give the same dS bit for bit.
template <int DK>
__device__ __forceinline__ void dS_step(const BwdSmem<DK> &s, const Lanes<DK> &L, float (&dS)[2][DK / 8], int tl) {
    constexpr int CW = DK / 8;
    const float gg = s.g[tl], bb = s.beta[tl];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float dyv = s.dy[tl][L.rl[i]];
        const float2 dy2 = make_float2(dyv, dyv);
        float2 dd01 = make_float2(0.0f, 0.0f), dd23 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < CW; j += 4) {
            const float2 a = __ffma2_rn(dy2, pair(s.q[tl], L.col(j)), pair(dS[i], j));
            const float2 c = __ffma2_rn(dy2, pair(s.q[tl], L.col(j + 2)), pair(dS[i], j + 2));
            dS[i][j] = a.x; dS[i][j + 1] = a.y; dS[i][j + 2] = c.x; dS[i][j + 3] = c.y;
            dd01 = __ffma2_rn(a, pair(s.k[tl], L.col(j)), dd01);
            dd23 = __ffma2_rn(c, pair(s.k[tl], L.col(j + 2)), dd23);
        }
        const float dd4[4] = {dd01.x, dd01.y, dd23.x, dd23.y};
        const float dd = row_sum(sum4(dd4));
        const float du = bb * dd;
        const float2 ndu2 = make_float2(-du, -du), g2 = make_float2(gg, gg);
#pragma unroll
        for (int j = 0; j < CW; j += 2) {
            const float2 r = __fmul2_rn(__ffma2_rn(ndu2, pair(s.k[tl], L.col(j)), pair(dS[i], j)), g2);
            dS[i][j] = r.x;
            dS[i][j + 1] = r.y;
        }
    }
}

// One full reverse step at tl of the chunk staged at t0: X holds the state
// after the step, Sp the state before it, dS the gradient of the state after
// it (returned as that of the state before it).  X is read first (for dq)
// and then reloaded with the state before step tl - 1 from the history, so
// two buffers in alternating roles carry the walk with no copies.  Adds the
// step's dq / dk column sums and dg / dbeta to the chunk's shared sums and
// writes dv.  Block-wide (the mask is uniform).
template <int DK>
__device__ __forceinline__ void reverse_step(const BwdParams &p, BwdSmem<DK> &s, const Lanes<DK> &L,
                                             const float *hist, int b, int hv, int r0, int t0, int tl,
                                             float (&X)[2][DK / 8], const float (&Sp)[2][DK / 8],
                                             float (&dS)[2][DK / 8]) {
    constexpr int CW = DK / 8;
    const bool live = s.m[tl] != 0;
    float dq_p[CW];
#pragma unroll
    for (int j = 0; j < CW; ++j) dq_p[j] = 0.0f;
    if (live) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float dyv = s.dy[tl][L.rl[i]];
#pragma unroll
            for (int j = 0; j < CW; ++j) dq_p[j] = fmaf(X[i][j], dyv, dq_p[j]);
        }
    }
    if (tl > 0) L.load(hist + (size_t)(tl - 1) * kRows * DK, X);
    if (!live) return;   // a masked step passes dS through
    const float gg = s.g[tl], bb = s.beta[tl];
    float dk_p[CW];
#pragma unroll
    for (int j = 0; j < CW; ++j) dk_p[j] = 0.0f;
    float dg_p = 0.0f, db_p = 0.0f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float dyv = s.dy[tl][L.rl[i]];
        const float ui = s.u[tl][L.rl[i]];
        float dd4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < CW; ++j) {
            dS[i][j] = fmaf(dyv, s.q[tl][L.col(j)], dS[i][j]);
            dd4[j & 3] = fmaf(dS[i][j], s.k[tl][L.col(j)], dd4[j & 3]);
        }
        const float dd = row_sum(sum4(dd4));    // ddelta of the row
        const float dl = bb * ui;               // delta
        const float du = bb * dd;
        const float ngdu = -gg * du;
        if (L.cg == 0) {
            db_p = fmaf(dd, ui, db_p);
            p.dv[(((size_t)b * p.T + t0 + tl) * p.Hv + hv) * p.Dv + r0 + L.rl[i]] = du;
        }
#pragma unroll
        for (int j = 0; j < CW; ++j) {
            dk_p[j] = fmaf(dS[i][j], dl, dk_p[j]);
            dS[i][j] = fmaf(-du, s.k[tl][L.col(j)], dS[i][j]);
            dk_p[j] = fmaf(Sp[i][j], ngdu, dk_p[j]);
            dg_p = fmaf(dS[i][j], Sp[i][j], dg_p);
            dS[i][j] *= gg;
        }
    }
    // sum the 2*CW partials (dq, dk) over the warp's four row groups in two
    // exchanges that halve the vector: lanes whose rg differs in bit 0 swap
    // halves (dq <-> dk), then lanes whose rg differs in bit 1 swap quarters,
    // so each lane ends with CW/2 summed columns (of dq for even rg, dk for
    // odd) and adds those; the pairwise sums are those of a per-column
    // shuffle sum
    const bool hi0 = (L.rg & 1) != 0, hi1 = (L.rg & 2) != 0;
    float h[CW];
#pragma unroll
    for (int j = 0; j < CW; ++j) {
        const float send = hi0 ? dq_p[j] : dk_p[j];
        const float keep = hi0 ? dk_p[j] : dq_p[j];
        h[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    constexpr int HQ = CW / 2;
    const int off = hi1 ? HQ : 0;
#pragma unroll
    for (int j = 0; j < HQ; ++j) {
        const float send = hi1 ? h[j] : h[HQ + j];
        const float keep = hi1 ? h[HQ + j] : h[j];
        const int c = L.col(off + j);
        atomicAdd(&s.red[tl][hi0 ? red_k<DK>(c) : red_q<DK>(c)], keep + __shfl_xor_sync(0xffffffffu, send, 16));
    }
    dg_p = warp_sum(dg_p);
    db_p = warp_sum(db_p);
    if (L.lane == 0) {
        atomicAdd(&s.red_g[tl], dg_p);
        atomicAdd(&s.red_b[tl], db_p);
    }
}

// The full reverse over the chunk of kC steps at t0 (at least one valid
// step): S is the state before it (clobbered), dS the gradient of the state
// after it, returned as the gradient of the state before it.  Recomputes the
// chunk's states into `hist` ([kC][kRows][DK]) and adds its gradients to the
// outputs.  Block-wide.
template <int DK>
__device__ __forceinline__ void reverse_chunk(const BwdParams &p, BwdSmem<DK> &s, const Lanes<DK> &L, float *hist,
                                           int b, int hk, int hv, int r0, int t0, float (&S)[2][DK / 8],
                                           float (&dS)[2][DK / 8]) {
    constexpr int CW = DK / 8;
    const int tid = threadIdx.x;
    const int T = p.T;
    stage_chunk<DK>(p, s, b, hk, hv, r0, t0, true);
    for (int i = tid; i < kC * DK; i += kThreads) {
        s.red[i / DK][red_q<DK>(i % DK)] = 0.0f;
        s.red[i / DK][red_k<DK>(i % DK)] = 0.0f;
    }
    if (tid < kC) {
        s.red_g[tid] = 0.0f;
        s.red_b[tid] = 0.0f;
    }
    // recompute the chunk: hist[tl] = the state before step tl
    for (int tl = 0; tl < kC; ++tl) {
        L.store(hist + (size_t)tl * kRows * DK, S);
        if (!s.m[tl]) continue;
        float u[2];
        fwd_step<DK>(s, L, S, tl, u);
        if (L.cg == 0) {
            s.u[tl][L.rl[0]] = u[0];
            s.u[tl][L.rl[1]] = u[1];
        }
    }
    __syncthreads();
    // S is now the state after the chunk; walk it backwards with S and Y in
    // alternating roles (see reverse_step), Y first the state before the
    // chunk's last step
    float Y[2][CW];
    L.load(hist + (size_t)(kC - 1) * kRows * DK, Y);
    static_assert(kC % 2 == 0, "the reverse walks the chunk in pairs of steps");
    for (int tl = kC - 1; tl >= 1; tl -= 2) {
        reverse_step<DK>(p, s, L, hist, b, hv, r0, t0, tl, S, Y, dS);
        reverse_step<DK>(p, s, L, hist, b, hv, r0, t0, tl - 1, Y, S, dS);
    }
    __syncthreads();
    // add the chunk's sums to the outputs (also summing over row slices
    // and over the v-heads of the k-head)
    // (four columns per reduction: they never straddle the skew at DK/2)
    const int n = min(kC, T - t0);
    for (int i = tid; i < n * (DK / 4); i += kThreads) {
        const int tl = i / (DK / 4), j = (i % (DK / 4)) * 4;
        if (!s.m[tl]) continue;
        const size_t o = (((size_t)b * T + t0 + tl) * p.Hk + hk) * DK + j;
        const float *rq = &s.red[tl][red_q<DK>(j)], *rk = &s.red[tl][red_k<DK>(j)];
        red_add_v4(p.dq + o, rq[0], rq[1], rq[2], rq[3]);
        red_add_v4(p.dk + o, rk[0], rk[1], rk[2], rk[3]);
    }
    if (tid < n && s.m[tid]) {
        const size_t o = ((size_t)b * T + t0 + tid) * p.Hv + hv;
        atomicAdd(p.dg + o, s.red_g[tid]);
        atomicAdd(p.dbeta + o, s.red_b[tid]);
    }
    __syncthreads();
}

// The forward direction over chunks [c_begin, c_end) of a row slice, S the
// initial state on entry and the final one on exit: stores S at the start of
// chunk c at ck + c * kRows * DK.  The next chunk's inputs are loaded into
// registers while the current one is stepped through.  Block-wide.
template <int DK>
__device__ __forceinline__ void forward_sweep(const BwdParams &p, BwdSmem<DK> &s, const Lanes<DK> &L, int b, int hk,
                                              int hv, int r0, int c_begin, int c_end, float *ck,
                                              float (&S)[2][DK / 8]) {
    if (c_begin >= c_end) return;
    ChunkRegs<DK> r;
    fetch_chunk<DK>(p, r, b, hk, hv, r0, c_begin * kC, false);
    for (int c = c_begin; c < c_end; ++c) {
        L.store(ck + (size_t)c * kRows * DK, S);
        commit_chunk<DK>(s, r);
        __syncthreads();
        if (c + 1 < c_end) fetch_chunk<DK>(p, r, b, hk, hv, r0, (c + 1) * kC, false);
        for (int tl = 0; tl < kC; ++tl) {
            if (!s.m[tl]) continue;   // a masked step is the identity on the state
            float u[2];
            fwd_step<DK>(s, L, S, tl, u);
        }
        __syncthreads();
    }
}

// Launch 1: per (row slice, head) a forward-sweep CTA (blockIdx.x < slices)
// storing S at the start of every chunk, and a reverse-sweep CTA storing dS
// at the end of every chunk and the gradient of the initial state.
template <int DK>
__global__ void __launch_bounds__(kThreads) bwd_sweep_kernel(const BwdParams p) {
    constexpr int CW = DK / 8;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<DK> &s = *reinterpret_cast<BwdSmem<DK> *>(smem_raw);
    const Lanes<DK> L;
    const int nsl = p.Dv / kRows;
    const bool reverse = (int)blockIdx.x >= nsl;
    const int slice = blockIdx.x % nsl, hv = blockIdx.y;
    const int b = p.order != nullptr ? p.order[blockIdx.z] : (int)blockIdx.z;
    const int hk = hv / (p.Hv / p.Hk);
    const int r0 = slice * kRows;
    const size_t head = (size_t)b * p.Hv + hv;
    const size_t rec = (head * nsl + slice) * (size_t)p.nck * kRows * DK;   // this slice's chunk records
    int c_begin, c_end;
    valid_chunks<DK>(p, s, b, c_begin, c_end);

    if (!reverse) {
        float S[2][CW];
        L.load_or_zero(p.state_in == nullptr ? nullptr : p.state_in + (head * p.Dv + r0) * DK, S);
        forward_sweep<DK>(p, s, L, b, hk, hv, r0, c_begin, c_end, p.ck + rec, S);
    } else {
        float dS[2][CW];
        L.load_or_zero(p.dstate_out == nullptr ? nullptr : p.dstate_out + (head * p.Dv + r0) * DK, dS);
        ChunkRegs<DK> r;
        if (c_begin < c_end) fetch_chunk<DK>(p, r, b, hk, hv, r0, (c_end - 1) * kC, true);
        for (int c = c_end - 1; c >= c_begin; --c) {
            L.store(p.dck + rec + (size_t)c * kRows * DK, dS);
            commit_chunk<DK>(s, r);
            __syncthreads();
            if (c > c_begin) fetch_chunk<DK>(p, r, b, hk, hv, r0, (c - 1) * kC, true);
            for (int tl = kC - 1; tl >= 0; --tl)
                if (s.m[tl]) dS_step<DK>(s, L, dS, tl);   // a masked step passes dS through
            __syncthreads();
        }
        L.store(p.dstate_in + (head * p.Dv + r0) * DK, dS);
    }
}

// Launch 2: every (chunk, row slice, head) item independently, CTA i taking
// items i, i + gridDim.x, ... with its own history buffer: the chunk's
// reverse from its S and its end dS.
template <int DK>
__global__ void __launch_bounds__(kThreads, 2) bwd_chunk_kernel(const BwdParams p, int n_items) {
    constexpr int CW = DK / 8;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<DK> &s = *reinterpret_cast<BwdSmem<DK> *>(smem_raw);
    const Lanes<DK> L;
    const int nsl = p.Dv / kRows;
    float *hist = p.hist + (size_t)blockIdx.x * kC * kRows * DK;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int c = item % p.nck;
        int rest = item / p.nck;
        const int slice = rest % nsl;
        rest /= nsl;
        const int hv = rest % p.Hv, b = rest / p.Hv;
        const int hk = hv / (p.Hv / p.Hk);
        const int r0 = slice * kRows;
        if (!chunk_active(p, b, c * kC)) continue;   // uniform: its gradients stay zero
        const size_t rec = ((((size_t)b * p.Hv + hv) * nsl + slice) * p.nck + c) * kRows * DK;
        float S[2][CW], dS[2][CW];
        L.load(p.dck + rec, dS);
        L.load(p.ck + rec, S);
        reverse_chunk<DK>(p, s, L, hist, b, hk, hv, r0, c * kC, S, dS);
    }
}

// Single launch for grids that fill the GPU on their own (at least two row
// slices per SM), where the split form only adds work: one CTA per (row
// slice, head) runs the forward sweep storing S at every chunk, then the
// chunks backwards with its own history buffer.
template <int DK>
__global__ void __launch_bounds__(kThreads, 2) bwd_fused_kernel(const BwdParams p) {
    constexpr int CW = DK / 8;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<DK> &s = *reinterpret_cast<BwdSmem<DK> *>(smem_raw);
    const Lanes<DK> L;
    const int nsl = p.Dv / kRows;
    const int slice = blockIdx.x, hv = blockIdx.y;
    const int b = p.order != nullptr ? p.order[blockIdx.z] : (int)blockIdx.z;
    const int hk = hv / (p.Hv / p.Hk);
    const int r0 = slice * kRows;
    const size_t head = (size_t)b * p.Hv + hv;
    const size_t cta = head * nsl + slice;
    float *ck = p.ck + cta * (size_t)p.nck * kRows * DK;
    float *hist = p.hist + cta * (size_t)kC * kRows * DK;
    int c_begin, c_end;
    valid_chunks<DK>(p, s, b, c_begin, c_end);

    float S[2][CW];
    L.load_or_zero(p.state_in == nullptr ? nullptr : p.state_in + (head * p.Dv + r0) * DK, S);
    forward_sweep<DK>(p, s, L, b, hk, hv, r0, c_begin, c_end, ck, S);
    float dS[2][CW];
    L.load_or_zero(p.dstate_out == nullptr ? nullptr : p.dstate_out + (head * p.Dv + r0) * DK, dS);
    for (int c = c_end - 1; c >= c_begin; --c) {
        if (!chunk_active(p, b, c * kC)) continue;   // dS passes through; its gradients stay zero
        L.load(ck + (size_t)c * kRows * DK, S);
        reverse_chunk<DK>(p, s, L, hist, b, hk, hv, r0, c * kC, S, dS);
    }
    L.store(p.dstate_in + (head * p.Dv + r0) * DK, dS);
}

// Workspace layout of either form: S at the start of every chunk (rec), the
// split form also dS at the end of every chunk (dck), and a history per CTA.
struct Layout {
    bool fused;
    int nsl, nck, items, slots;
    size_t rec_floats, dck_floats, hist_floats;
};

Layout layout_of(const Sizes &s) {
    Layout l;
    l.nsl = s.Dv / kRows;
    l.nck = (s.T + kC - 1) / kC;
    const long slices = (long)s.B * s.Hv * l.nsl;
    l.fused = slices >= 2L * num_sms();
    l.rec_floats = (size_t)slices * l.nck * kRows * s.Dk;
    if (l.fused) {
        l.items = 0;
        l.slots = (int)slices;
        l.dck_floats = 0;
    } else {
        const long items = slices * l.nck;
        l.items = (int)items;
        l.slots = (int)std::min<long>(items, 2L * num_sms());
        l.dck_floats = l.rec_floats;
    }
    l.hist_floats = (size_t)l.slots * kC * kRows * s.Dk;
    return l;
}

template <int DK>
cudaError_t launch_bwd_t(const Sizes &s, const Layout &l, const BwdParams &p, cudaStream_t st) {
    const size_t smem = sizeof(BwdSmem<DK>);
    static unsigned long long done_sweep = 0, done_chunk = 0, done_fused = 0;   // per instantiation, per device
    cudaError_t e = set_max_smem(done_sweep, bwd_sweep_kernel<DK>, smem);
    if (e == cudaSuccess) e = set_max_smem(done_chunk, bwd_chunk_kernel<DK>, smem);
    if (e == cudaSuccess) e = set_max_smem(done_fused, bwd_fused_kernel<DK>, smem);
    if (e != cudaSuccess) return e;
    if (l.fused) {
        bwd_fused_kernel<DK><<<dim3(l.nsl, s.Hv, s.B), kThreads, smem, st>>>(p);
        return cudaGetLastError();
    }
    bwd_sweep_kernel<DK><<<dim3(2 * l.nsl, s.Hv, s.B), kThreads, smem, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess || l.items == 0) return e;
    bwd_chunk_kernel<DK><<<l.slots, kThreads, smem, st>>>(p, l.items);
    return cudaGetLastError();
}

}  // namespace

size_t backward_workspace(const Sizes &s) {
    const Layout l = layout_of(s);
    return row_order_workspace(s) + (l.rec_floats + l.dck_floats + l.hist_floats) * sizeof(float);
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
    const Layout l = layout_of(s);
    if (!l.fused && (long)s.B * s.Hv * l.nsl * l.nck > (long)INT_MAX) return cudaErrorNotSupported;   // item index
    // rows longest first (the row order's scratch, a multiple of 256 bytes,
    // leads the workspace)
    const int *order = nullptr;
    if (mask != nullptr && s.B > 1) {
        e = launch_row_order(s, mask, ws, st);
        if (e != cudaSuccess) return e;
        order = static_cast<const int *>(ws);
    }
    float *ck = reinterpret_cast<float *>(static_cast<char *>(ws) + row_order_workspace(s));
    float *dck = ck + l.rec_floats;
    float *hist = dck + l.dck_floats;
    BwdParams p{q, k, v, g, beta, state_in, mask, dy, dstate_out, dq, dk, dv, dg, dbeta, dstate_in,
                ck, dck, hist, order, s.B, s.T, s.Hk, s.Hv, s.Dv, l.nck};
    switch (s.Dk) {
        case 32: return launch_bwd_t<32>(s, l, p, st);
        case 64: return launch_bwd_t<64>(s, l, p, st);
        case 128: return launch_bwd_t<128>(s, l, p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
