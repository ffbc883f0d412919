/*
 * ssm_oracle.c -- plain sequential fp64 CPU oracle for the Mamba-1 selective scan.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's CPU
 * baseline may load this library. It shares no code, header, table or helper
 * with the CUDA path in selective_state_space_121_b300/.
 *
 * What it computes follows the pages:
 *   - Mamba SSM complete guide (youngju.dev), section 5, "complete Mamba
 *     implementation", MambaBlock.selective_scan: per step
 *         x <- exp(delta*A) * x + delta*B*u ;  y = <x, C> ;  y += u*D
 *     (the discretised recurrence of section 2, "Discretization", with the
 *     simplified input matrix delta*B that the page's selective_scan uses);
 *   - same page, MambaBlock.ssm: delta = softplus(dt_proj(...)), where the
 *     dt_proj bias is the per-channel delta_bias added before the softplus;
 *   - same page, MambaBlock.forward: y = y * silu(z) after the scan.
 * The state starts at h0 (zero when absent), as in the SM1 page's closed form
 * which carries an h0 (Scalar Mamba1 page (aitrends.kr), section details).
 *
 * Readings where the pages are silent: softplus is PyTorch's default
 * (beta = 1, the identity above 20); silu(z) = z / (1 + exp(-z)).
 *
 * Inputs are the exact stored values (bf16 values widened exactly to fp32) and
 * are widened to double here; every operation runs in double, in the order the
 * page's loop runs it (n ascending inside each step). Channels (b, d) are
 * independent, so the OpenMP loop over channels does not change any result.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

double oracle_softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }

double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* Layouts (row-major, last index fastest):
 *   u, delta, z : (batch, dim, seqlen)      y      : (batch, dim, seqlen)
 *   B, C        : (batch, dstate, seqlen)   h0     : (batch, dim, dstate) or NULL
 *   A           : (dim, dstate)             h_last : (batch, dim, dstate) or NULL
 *   D, delta_bias : (dim) or NULL           z      : NULL when not gated
 * Returns 0, or -1 on a bad size.
 */
int oracle_scan(const float *u, const float *delta, const float *A, const float *B,
                const float *C, const float *D, const float *z, const float *delta_bias,
                int softplus, const double *h0, double *y, double *h_last, int64_t batch,
                int64_t dim, int64_t seqlen, int64_t dstate, int nthreads) {
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1) return -1;
    int64_t nch = batch * dim;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (int64_t ch = 0; ch < nch; ch++) {
        int64_t b = ch / dim, d = ch % dim;
        double *h = (double *)malloc(sizeof(double) * (size_t)dstate);
        for (int64_t n = 0; n < dstate; n++) h[n] = h0 ? h0[ch * dstate + n] : 0.0;
        const float *u_r = u + ch * seqlen, *dl_r = delta + ch * seqlen;
        const float *z_r = z ? z + ch * seqlen : NULL;
        const float *B_b = B + b * dstate * seqlen, *C_b = C + b * dstate * seqlen;
        const float *A_d = A + d * dstate;
        for (int64_t t = 0; t < seqlen; t++) {
            double ut = (double)u_r[t];
            double x = (double)dl_r[t] + (delta_bias ? (double)delta_bias[d] : 0.0);
            double dt = softplus ? oracle_softplus(x) : x;
            double acc = 0.0;
            for (int64_t n = 0; n < dstate; n++) {
                double a = exp(dt * (double)A_d[n]);
                double bu = dt * (double)B_b[n * seqlen + t] * ut;
                h[n] = a * h[n] + bu;
                acc += (double)C_b[n * seqlen + t] * h[n];
            }
            double yv = acc + (D ? (double)D[d] * ut : 0.0);
            if (z_r) yv *= oracle_silu((double)z_r[t]);
            y[ch * seqlen + t] = yv;
        }
        if (h_last)
            for (int64_t n = 0; n < dstate; n++) h_last[ch * dstate + n] = h[n];
        free(h);
    }
    return 0;
}

/* One decode token, in place on the fp64 state: the body of the same loop
 * applied once (the O(1)-per-token recurrent form).
 *   state : (batch, dim, dstate) in/out     x, delta, z, y : (batch, dim)
 *   B, C  : (batch, dstate)                 A : (dim, dstate); D, delta_bias : (dim)
 */
int oracle_state_update(double *state, const float *x, const float *delta, const float *A,
                        const float *B, const float *C, const float *D, const float *z,
                        const float *delta_bias, int softplus, double *y, int64_t batch,
                        int64_t dim, int64_t dstate, int nthreads) {
    if (batch < 0 || dim < 0 || dstate < 1) return -1;
    int64_t nch = batch * dim;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t ch = 0; ch < nch; ch++) {
        int64_t b = ch / dim, d = ch % dim;
        double xt = (double)x[ch];
        double v = (double)delta[ch] + (delta_bias ? (double)delta_bias[d] : 0.0);
        double dt = softplus ? oracle_softplus(v) : v;
        double acc = 0.0;
        double *s = state + ch * dstate;
        for (int64_t n = 0; n < dstate; n++) {
            double a = exp(dt * (double)A[d * dstate + n]);
            s[n] = a * s[n] + dt * (double)B[b * dstate + n] * xt;
            acc += (double)C[b * dstate + n] * s[n];
        }
        double yv = acc + (D ? (double)D[d] * xt : 0.0);
        if (z) yv *= oracle_silu((double)z[ch]);
        y[ch] = yv;
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
