/*
 * KDA recurrence oracle: plain, slow, sequential, fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link or call
 * this file; it exists so the tests, the smoke check and the benchmark's CPU
 * baseline can compare the CUDA kernels against an obviously correct
 * statement of the method.  It shares no code with the CUDA path.
 *
 * What it computes ("Colibri Kimi K3 Metal backend", architecture section:
 * the per-head delta-rule state update; section 8.2: the two-pass token step
 * whose second pass reads the output from the UPDATED state), per head, for
 * each token t in order:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * written out as the pages' two passes:
 *     a_i  = exp(g_i)                     (per-channel decay, section 8.4:
 *                                          alpha is per element, beta per head)
 *     S_ij = a_i * S_ij                   (row decay, pass 1)
 *     u_j  = sum_i k_i S_ij               (the "kS" column sums, pass 1)
 *     w_j  = beta * (v_j - u_j)           (the "vt" delta, pass 1)
 *     S_ij = S_ij + k_i w_j               (rank-1 update, pass 2)
 *     o_j  = sum_i q_i S_ij               (readout, pass 2)
 *
 * Expanding (I - beta k k^T) D S + beta k v^T = D S + k (beta (v - (D S)^T k))^T
 * shows the passes are the formula.  State layout S[i][j]: i the key channel
 * (dk), j the value channel (dv), row-major.  Inputs are upcast exactly to
 * double (bf16 bit patterns or fp32); all arithmetic is double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* kind: 0 fp32, 1 bf16 bit patterns, 2 double (already exact) */
static double load_in(const void *p, int is_bf16, int64_t idx)
{
    if (is_bf16 == 2)
        return ((const double *)p)[idx];
    if (is_bf16) {
        uint16_t b = ((const uint16_t *)p)[idx];
        uint32_t bits = ((uint32_t)b) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)p)[idx];
}

/*
 * One (sequence, head) unit over tokens [t0, t1) of a packed [T, H, d] batch.
 *   q, k      : [T, H, dk]   (qkv_bf16: 0 fp32, 1 bf16 bits, 2 double)
 *   v         : [T, H, dv]
 *   g         : [T, H, dk]   fp32 log-decay
 *   beta      : [T, H]       fp32
 *   S0        : [dk, dv]     double initial state of this unit (the caller upcasts
 *               an fp32 state exactly), or NULL (zeros)
 *   o_out     : [t1-t0, dv]  double, row r is token t0+r
 *   S_out     : [dk, dv]     double final state
 * Returns 0, or -1 if scratch allocation failed.
 */
int oracle_kda_unit(const void *q, const void *k, const void *v, int qkv_bf16,
                    const float *g, const float *beta, const double *S0,
                    int64_t t0, int64_t t1, int H, int h, int dk, int dv,
                    double *o_out, double *S_out)
{
    double *S = S_out;
    double *a = (double *)malloc(sizeof(double) * (size_t)dk);
    double *kk = (double *)malloc(sizeof(double) * (size_t)dk);
    double *qq = (double *)malloc(sizeof(double) * (size_t)dk);
    double *u = (double *)malloc(sizeof(double) * (size_t)dv);
    double *w = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!a || !kk || !qq || !u || !w) {
        free(a); free(kk); free(qq); free(u); free(w);
        return -1;
    }
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            S[(size_t)i * dv + j] = S0 ? S0[(size_t)i * dv + j] : 0.0;

    for (int64_t t = t0; t < t1; ++t) {
        const int64_t rk = (t * H + h) * (int64_t)dk;   /* row of q, k, g */
        const int64_t rv = (t * H + h) * (int64_t)dv;   /* row of v */
        const double b = (double)beta[t * H + h];
        for (int i = 0; i < dk; ++i) {
            a[i] = exp((double)g[rk + i]);
            kk[i] = load_in(k, qkv_bf16, rk + i);
            qq[i] = load_in(q, qkv_bf16, rk + i);
        }
        /* pass 1: decay the rows, then u = S^T k */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                S[(size_t)i * dv + j] *= a[i];
        for (int j = 0; j < dv; ++j)
            u[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                u[j] += kk[i] * S[(size_t)i * dv + j];
        for (int j = 0; j < dv; ++j)
            w[j] = b * (load_in(v, qkv_bf16, rv + j) - u[j]);
        /* pass 2: rank-1 update, then o = S^T q with the updated state */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                S[(size_t)i * dv + j] += kk[i] * w[j];
        double *o = o_out + (size_t)(t - t0) * dv;
        for (int j = 0; j < dv; ++j)
            o[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                o[j] += qq[i] * S[(size_t)i * dv + j];
    }
    free(a); free(kk); free(qq); free(u); free(w);
    return 0;
}

/*
 * One decode token for unit (b, h) of a [B, H, d] batch: the same update as
 * above applied once, starting from S_in ([dk, dv], upcast by the caller).
 */
int oracle_kda_decode_unit(const void *q, const void *k, const void *v, int qkv_bf16,
                           const float *g, const float *beta, const double *S_in,
                           int H, int b, int h, int dk, int dv,
                           double *o_out, double *S_out)
{
    return oracle_kda_unit(q, k, v, qkv_bf16, g, beta, S_in, (int64_t)b, (int64_t)b + 1,
                           H, h, dk, dv, o_out, S_out);
}
