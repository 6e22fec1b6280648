/*
 * CPU oracle for the gated delta-rule recurrence -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this file's shared library.  It shares no code, header or constant with the
 * CUDA library; it is the plain definition, in double precision, sequential in
 * t, with no blocking, fusion or reordering.
 *
 * Definition followed (one (b, hv) head at a time):
 *   "mlex 0.1.2, src/models/gated_delta.rs", GatedDeltaNet::forward, the
 *   per-timestep loop: the state is decayed by g_t, kv_mem = S k_t is read from
 *   the decayed state, delta = beta_t (v_t - kv_mem), S += delta k_t^T, and the
 *   output y_t = S q_t is read from the updated state.
 *   "mlx-bun 0.4.0 -> 1.0.0, package/src/model/qwen3-delta.ts", the
 *   gated_delta_step kernel source and its masked specialization (getKernel):
 *   a step whose mask is zero writes y = 0 and leaves the state untouched.
 *
 * Layouts (row-major, contiguous, all double except the mask):
 *   q, k [T, Dk]   v, y [T, Dv]   g, beta [T]   mask [T] (NULL = all valid)
 *   S [Dv, Dk], in/out: row i is output channel i, contiguous over Dk.
 */
#include <stddef.h>
#include <stdint.h>

void oracle_delta_rule_head(int T, int Dk, int Dv,
                            const double *q, const double *k, const double *v,
                            const double *g, const double *beta,
                            const uint8_t *mask, double *S, double *y)
{
    for (int t = 0; t < T; ++t) {
        const double *qt = q + (size_t)t * Dk;
        const double *kt = k + (size_t)t * Dk;
        const double *vt = v + (size_t)t * Dv;
        double *yt = y + (size_t)t * Dv;
        if (mask != NULL && mask[t] == 0) {
            for (int i = 0; i < Dv; ++i) yt[i] = 0.0;
            continue;
        }
        /* S <- g_t S */
        for (int i = 0; i < Dv; ++i)
            for (int j = 0; j < Dk; ++j) S[(size_t)i * Dk + j] *= g[t];
        /* per row i: kv = S_i . k_t ; delta = beta_t (v_i - kv) ; S_i += delta k_t */
        for (int i = 0; i < Dv; ++i) {
            double *Si = S + (size_t)i * Dk;
            double kv = 0.0;
            for (int j = 0; j < Dk; ++j) kv += Si[j] * kt[j];
            double delta = beta[t] * (vt[i] - kv);
            for (int j = 0; j < Dk; ++j) Si[j] += delta * kt[j];
        }
        /* y_t = S q_t (updated state) */
        for (int i = 0; i < Dv; ++i) {
            const double *Si = S + (size_t)i * Dk;
            double acc = 0.0;
            for (int j = 0; j < Dk; ++j) acc += Si[j] * qt[j];
            yt[i] = acc;
        }
    }
}

/*
 * Vectorized gating: the decay is one factor per key channel, g [T, Dk]
 * (the variant the qwen3-delta.ts page names beside the scalar one):
 *   S <- S diag(g_t), then the same kv_mem / delta / update / output steps.
 */
void oracle_delta_rule_head_vec(int T, int Dk, int Dv,
                                const double *q, const double *k, const double *v,
                                const double *g, const double *beta,
                                const uint8_t *mask, double *S, double *y)
{
    for (int t = 0; t < T; ++t) {
        const double *qt = q + (size_t)t * Dk;
        const double *kt = k + (size_t)t * Dk;
        const double *vt = v + (size_t)t * Dv;
        const double *gt = g + (size_t)t * Dk;
        double *yt = y + (size_t)t * Dv;
        if (mask != NULL && mask[t] == 0) {
            for (int i = 0; i < Dv; ++i) yt[i] = 0.0;
            continue;
        }
        /* S <- S diag(g_t): column j scaled by g_t[j] */
        for (int i = 0; i < Dv; ++i)
            for (int j = 0; j < Dk; ++j) S[(size_t)i * Dk + j] *= gt[j];
        for (int i = 0; i < Dv; ++i) {
            double *Si = S + (size_t)i * Dk;
            double kv = 0.0;
            for (int j = 0; j < Dk; ++j) kv += Si[j] * kt[j];
            double delta = beta[t] * (vt[i] - kv);
            for (int j = 0; j < Dk; ++j) Si[j] += delta * kt[j];
        }
        for (int i = 0; i < Dv; ++i) {
            const double *Si = S + (size_t)i * Dk;
            double acc = 0.0;
            for (int j = 0; j < Dk; ++j) acc += Si[j] * qt[j];
            yt[i] = acc;
        }
    }
}
