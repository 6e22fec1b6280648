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
#include <stdlib.h>
#include <string.h>

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

/*
 * Backward pass of oracle_delta_rule_head: the gradient of the recurrence
 * with respect to every input, given the gradient dy [T, Dv] of the outputs
 * and dST [Dv, Dk] of the final state (NULL = 0).  The pages define the
 * forward recurrence only; this is its exact derivative, taken step by step
 * in reverse.  With S' = g_t S_{t-1}, u = v_t - S' k_t, delta = beta_t u,
 * S_t = S' + delta k_t^T, y_t = S_t q_t, and dS the gradient of S_t:
 *   dS += dy_t q_t^T            dq_t = S_t^T dy_t
 *   ddelta = dS k_t             dk_t = dS^T delta
 *   dbeta_t = ddelta . u        du = beta_t ddelta        dv_t = du
 *   dS' = dS - du k_t^T         dk_t -= S'^T du
 *   dg_t = <dS', S_{t-1}>       dS_{t-1} = g_t dS'
 * A masked step has zero gradients for its inputs and passes dS through.
 * The forward states are recomputed and kept (T + 1 of them): fine for the
 * small cases the oracle serves.  Outputs: dq, dk [T, Dk], dv [T, Dv],
 * dg, dbeta [T], dS0 [Dv, Dk] (all written).
 */
int oracle_delta_rule_head_bwd(int T, int Dk, int Dv,
                               const double *q, const double *k, const double *v,
                               const double *g, const double *beta, const uint8_t *mask,
                               const double *S0, const double *dy, const double *dST,
                               double *dq, double *dk, double *dv, double *dg, double *dbeta,
                               double *dS0)
{
    const size_t n = (size_t)Dv * Dk;
    double *hist = (double *)malloc(sizeof(double) * n * (size_t)(T + 1));   /* S_{-1} .. S_{T-1} */
    double *u = (double *)malloc(sizeof(double) * (size_t)T * Dv);
    double *dS = (double *)malloc(sizeof(double) * n);
    double *Sp = (double *)malloc(sizeof(double) * n);
    double *ddel = (double *)malloc(sizeof(double) * (size_t)Dv);
    double *du = (double *)malloc(sizeof(double) * (size_t)Dv);
    if (!hist || !u || !dS || !Sp || !ddel || !du) {
        free(hist); free(u); free(dS); free(Sp); free(ddel); free(du);
        return -1;
    }
    /* forward, keeping every state: hist[t + 1] = S_t, hist[0] = S0 */
    for (size_t e = 0; e < n; ++e) hist[e] = S0 ? S0[e] : 0.0;
    for (int t = 0; t < T; ++t) {
        const double *prev = hist + (size_t)t * n;
        double *cur = hist + (size_t)(t + 1) * n;
        const double *kt = k + (size_t)t * Dk;
        const double *vt = v + (size_t)t * Dv;
        if (mask != NULL && mask[t] == 0) {
            memcpy(cur, prev, sizeof(double) * n);
            for (int i = 0; i < Dv; ++i) u[(size_t)t * Dv + i] = 0.0;
            continue;
        }
        for (int i = 0; i < Dv; ++i) {
            double kv = 0.0;
            for (int j = 0; j < Dk; ++j) kv += g[t] * prev[(size_t)i * Dk + j] * kt[j];
            const double ui = vt[i] - kv;
            u[(size_t)t * Dv + i] = ui;
            for (int j = 0; j < Dk; ++j)
                cur[(size_t)i * Dk + j] = g[t] * prev[(size_t)i * Dk + j] + beta[t] * ui * kt[j];
        }
    }
    /* reverse */
    for (size_t e = 0; e < n; ++e) dS[e] = dST ? dST[e] : 0.0;
    for (int t = T - 1; t >= 0; --t) {
        const double *St = hist + (size_t)(t + 1) * n;
        const double *Sprev = hist + (size_t)t * n;
        const double *qt = q + (size_t)t * Dk;
        const double *kt = k + (size_t)t * Dk;
        const double *dyt = dy + (size_t)t * Dv;
        double *dqt = dq + (size_t)t * Dk;
        double *dkt = dk + (size_t)t * Dk;
        double *dvt = dv + (size_t)t * Dv;
        for (int j = 0; j < Dk; ++j) { dqt[j] = 0.0; dkt[j] = 0.0; }
        for (int i = 0; i < Dv; ++i) dvt[i] = 0.0;
        dg[t] = 0.0;
        dbeta[t] = 0.0;
        if (mask != NULL && mask[t] == 0) continue;
        /* from y_t = S_t q_t */
        for (int i = 0; i < Dv; ++i)
            for (int j = 0; j < Dk; ++j) {
                dS[(size_t)i * Dk + j] += dyt[i] * qt[j];
                dqt[j] += St[(size_t)i * Dk + j] * dyt[i];
            }
        /* from S_t = S' + delta k_t^T */
        for (int i = 0; i < Dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < Dk; ++j) acc += dS[(size_t)i * Dk + j] * kt[j];
            ddel[i] = acc;
            const double delta = beta[t] * u[(size_t)t * Dv + i];
            for (int j = 0; j < Dk; ++j) dkt[j] += dS[(size_t)i * Dk + j] * delta;
        }
        /* from delta = beta_t u, u = v_t - S' k_t */
        for (int i = 0; i < Dv; ++i) {
            dbeta[t] += ddel[i] * u[(size_t)t * Dv + i];
            du[i] = beta[t] * ddel[i];
            dvt[i] = du[i];
        }
        for (size_t e = 0; e < n; ++e) Sp[e] = g[t] * Sprev[e];
        for (int i = 0; i < Dv; ++i)
            for (int j = 0; j < Dk; ++j) {
                dS[(size_t)i * Dk + j] -= du[i] * kt[j];
                dkt[j] -= Sp[(size_t)i * Dk + j] * du[i];
            }
        /* from S' = g_t S_{t-1} */
        double acc = 0.0;
        for (size_t e = 0; e < n; ++e) acc += dS[e] * Sprev[e];
        dg[t] = acc;
        for (size_t e = 0; e < n; ++e) dS[e] *= g[t];
    }
    for (size_t e = 0; e < n; ++e) dS0[e] = dS[e];
    free(hist); free(u); free(dS); free(Sp); free(ddel); free(du);
    return 0;
}
