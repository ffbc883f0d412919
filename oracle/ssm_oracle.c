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

/* The same selective scan along another traversal of the sequence, with the
 * exact zero-order-hold input matrix as an option.
 *
 * Traversal (Mamba SSM complete guide, section 9 "Mamba applications", VMamba:
 * an image of rows x cols patches, stored in raster order, is scanned in four
 * directions). Step k = 0 .. seqlen-1 of the scan visits position pos(k):
 *   order 0  raster             pos(k) = k
 *   order 1  reversed raster    pos(k) = seqlen - 1 - k
 *   order 2  column-major       pos(k) = (k % rows) * cols + k / rows
 *   order 3  reversed columns   pos(k) = column-major pos(seqlen - 1 - k)
 * (rows * cols == seqlen for orders 2 and 3). Every input is read at pos(k)
 * and the step's output is written to y at pos(k): each direction's output
 * lands in raster order. h0 is the state before the first visited step,
 * h_last the state after the last.
 *
 * Input matrix. zoh == 0: dt * B (the selective_scan form, as oracle_scan).
 * zoh != 0: the zero-order hold of the same guide's section 2
 * ("Discretization"), B_bar = (dt A)^-1 (exp(dt A) - 1) dt B, which for the
 * diagonal A of the scan is (exp(dt A) - 1) / A * B, and dt * B where A = 0.
 * Layouts and other arguments as oracle_scan.
 */
static int64_t oracle_pos(int order, int64_t k, int64_t L, int64_t rows, int64_t cols) {
    if (order == 1 || order == 3) k = L - 1 - k;
    if (order >= 2) return (k % rows) * cols + k / rows;
    return k;
}

int oracle_scan_dir(const float *u, const float *delta, const float *A, const float *B,
                    const float *C, const float *D, const float *z, const float *delta_bias,
                    int softplus, const double *h0, double *y, double *h_last, int64_t batch,
                    int64_t dim, int64_t seqlen, int64_t dstate, int order, int64_t rows,
                    int64_t cols, int zoh, int nthreads) {
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1 || order < 0 || order > 3) return -1;
    if (order >= 2 && (rows < 1 || cols < 1 || rows * cols != seqlen)) return -1;
    int64_t nch = batch * dim;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (int64_t ch = 0; ch < nch; ch++) {
        int64_t b = ch / dim, d = ch % dim;
        double *h = (double *)malloc(sizeof(double) * (size_t)dstate);
        const double *h0_r = h0 ? h0 + ch * dstate : NULL;
        for (int64_t n = 0; n < dstate; n++) h[n] = h0_r ? h0_r[n] : 0.0;
        const float *u_r = u + ch * seqlen, *dl_r = delta + ch * seqlen;
        const float *z_r = z ? z + ch * seqlen : NULL;
        const float *B_b = B + b * dstate * seqlen, *C_b = C + b * dstate * seqlen;
        const float *A_row = A + d * dstate;
        for (int64_t k = 0; k < seqlen; k++) {
            int64_t t = oracle_pos(order, k, seqlen, rows, cols);
            double ut = (double)u_r[t];
            double v = (double)dl_r[t];
            if (delta_bias) v += (double)delta_bias[d];
            double dt = softplus ? oracle_softplus(v) : v;
            double acc = 0.0;
            for (int64_t n = 0; n < dstate; n++) {
                double an = (double)A_row[n];
                double a = exp(dt * an);
                double bbar = zoh ? (an != 0.0 ? expm1(dt * an) / an : dt) : dt;
                h[n] = a * h[n] + bbar * (double)B_b[n * seqlen + t] * ut;
                acc += (double)C_b[n * seqlen + t] * h[n];
            }
            if (D) acc += (double)D[d] * ut;
            if (z_r) acc *= oracle_silu((double)z_r[t]);
            y[ch * seqlen + t] = acc;
        }
        if (h_last) {
            double *hl_r = h_last + ch * dstate;
            for (int64_t n = 0; n < dstate; n++) hl_r[n] = h[n];
        }
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

/* Backward of oracle_scan: the gradients of a loss l(out, h_last) given
 * dout = dl/dout (batch, dim, seqlen) and dh_last = dl/dh_last (or NULL), by the
 * chain rule through the same operations in reverse (the pages print no
 * backward; this is the derivative of the forward above, step by step):
 *   out_t = y_t silu(z_t),  y_t = sum_n C_tn h_tn + D u_t,
 *   h_tn = a_tn h_{t-1,n} + dt_t B_tn u_t,  a_tn = exp(dt_t A_n),
 *   dt_t = softplus(delta_t + bias) (or the raw sum).
 * With g_n = dl/dh_tn accumulated backwards (g starts at dh_last):
 *   dy = dout silu(z); dz = dout y silu'(z), silu'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *   g_n += C_tn dy;  dC_tn += dy h_tn;  dD += dy u;  du += D dy
 *   d(dt) += sum_n g_n (h_{t-1,n} a_tn A_n + B_tn u);  dA_n += g_n h_{t-1,n} a_tn dt
 *   dB_tn += g_n dt u;  du += sum_n g_n dt B_tn;  then g_n *= a_tn
 *   ddelta = d(dt) sigmoid(delta + bias) (softplus' ; 1 without softplus, and the
 *   identity branch above 20); dbias += ddelta;  finally dh0 = g.
 * Sums over channels (dB, dC) run in channel order inside each batch row (rows
 * in parallel); sums over batch rows (dA, dD, dbias) in a fixed order after.
 *   du, ddelta, dz : (batch, dim, seqlen)   dB, dC : (batch, dstate, seqlen)
 *   dA : (dim, dstate)   dD, dbias : (dim)   dh0 : (batch, dim, dstate)
 * dz may be NULL when z is; the others are required. */
int oracle_scan_bwd(const float *u, const float *delta, const float *A, const float *B,
                    const float *C, const float *D, const float *z, const float *delta_bias,
                    int softplus, const double *h0, const double *dout, const double *dh_last,
                    double *du, double *ddelta, double *dA, double *dB, double *dC, double *dD,
                    double *dz, double *dbias, double *dh0, int64_t batch, int64_t dim,
                    int64_t seqlen, int64_t dstate, int nthreads) {
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1) return -1;
    int64_t nch = batch * dim, N = dstate, L = seqlen;
    /* per-channel partials of the sums over batch rows, reduced afterwards */
    double *pA = (double *)calloc((size_t)(nch * N) + 1, sizeof(double));
    double *pD = (double *)calloc((size_t)nch + 1, sizeof(double));
    double *pbias = (double *)calloc((size_t)nch + 1, sizeof(double));
    if (!pA || !pD || !pbias) return -2;
    for (int64_t k = 0; k < batch * N * L; k++) { dB[k] = 0.0; dC[k] = 0.0; }
    /* batch rows in parallel; inside a row the channels run in order d = 0, 1, ...
     * and add their dB, dC contributions directly (the sum over channels) */
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t b = 0; b < batch; b++) {
        double *hs = (double *)malloc(sizeof(double) * (size_t)((L + 1) * N));
        double *g = (double *)malloc(sizeof(double) * (size_t)N);
        const float *B_b = B + b * N * L, *C_b = C + b * N * L;
        double *dB_b = dB + b * N * L, *dC_b = dC + b * N * L;
        for (int64_t d = 0; d < dim; d++) {
            int64_t ch = b * dim + d;
            const float *u_r = u + ch * L, *dl_r = delta + ch * L;
            const float *z_r = z ? z + ch * L : NULL;
            const float *A_d = A + d * N;
            double bias = delta_bias ? (double)delta_bias[d] : 0.0;
            double Dd = D ? (double)D[d] : 0.0;
            /* forward, keeping every state: hs[(t + 1) * N + n] = h_tn, hs[n] = h0 */
            for (int64_t n = 0; n < N; n++) hs[n] = h0 ? h0[ch * N + n] : 0.0;
            for (int64_t t = 0; t < L; t++) {
                double x = (double)dl_r[t] + bias;
                double dt = softplus ? oracle_softplus(x) : x;
                for (int64_t n = 0; n < N; n++)
                    hs[(t + 1) * N + n] = exp(dt * (double)A_d[n]) * hs[t * N + n] +
                                          dt * (double)B_b[n * L + t] * (double)u_r[t];
            }
            for (int64_t n = 0; n < N; n++) g[n] = dh_last ? dh_last[ch * N + n] : 0.0;
            for (int64_t t = L - 1; t >= 0; t--) {
                double ut = (double)u_r[t];
                double x = (double)dl_r[t] + bias;
                double dt = softplus ? oracle_softplus(x) : x;
                double yv = Dd * ut;
                for (int64_t n = 0; n < N; n++) yv += (double)C_b[n * L + t] * hs[(t + 1) * N + n];
                double dy = dout[ch * L + t];
                if (z_r) {
                    double zz = (double)z_r[t];
                    double sg = 1.0 / (1.0 + exp(-zz));
                    dz[ch * L + t] = dy * yv * sg * (1.0 + zz * (1.0 - sg));
                    dy *= zz * sg;
                } else if (dz) {
                    dz[ch * L + t] = 0.0;
                }
                pD[ch] += dy * ut;
                double dut = Dd * dy, ddt = 0.0;
                for (int64_t n = 0; n < N; n++) {
                    double Cn = (double)C_b[n * L + t], Bn = (double)B_b[n * L + t];
                    double an = exp(dt * (double)A_d[n]);
                    double hprev = hs[t * N + n];
                    g[n] += Cn * dy;
                    dC_b[n * L + t] += dy * hs[(t + 1) * N + n];
                    ddt += g[n] * (hprev * an * (double)A_d[n] + Bn * ut);
                    pA[ch * N + n] += g[n] * hprev * an * dt;
                    dB_b[n * L + t] += g[n] * dt * ut;
                    dut += g[n] * dt * Bn;
                    g[n] *= an;
                }
                double dx = ddt;
                if (softplus) dx = x > 20.0 ? ddt : ddt / (1.0 + exp(-x));
                du[ch * L + t] = dut;
                ddelta[ch * L + t] = dx;
                pbias[ch] += dx;
            }
            for (int64_t n = 0; n < N; n++) dh0[ch * N + n] = g[n];
        }
        free(hs);
        free(g);
    }
    for (int64_t d = 0; d < dim; d++) {
        double sD = 0.0, sb = 0.0;
        for (int64_t b = 0; b < batch; b++) {
            sD += pD[b * dim + d];
            sb += pbias[b * dim + d];
        }
        dD[d] = sD;
        dbias[d] = sb;
        for (int64_t n = 0; n < N; n++) {
            double sA = 0.0;
            for (int64_t b = 0; b < batch; b++) sA += pA[(b * dim + d) * N + n];
            dA[d * N + n] = sA;
        }
    }
    free(pA); free(pD); free(pbias);
    return 0;
}

/* Mamba-2 multi-head SSM (the next row after the Mamba-1 path; Mamba SSM complete
 * guide (youngju.dev), section 6 "Mamba 2": a scalar A per head, the state of a
 * head a (headdim x dstate) matrix, heads grouped over shared B and C), written as
 * its defining recurrence, sequentially in fp64:
 *     dt = softplus(dt_raw + dt_bias_h)                (raw sum without softplus)
 *     H_t = exp(dt A_h) H_{t-1} + dt x_t B_t^T,   y_t = H_t C_t + D_h x_t,   y_t *= silu(z_t)
 * Readings where the page gives no code (its Mamba2Block.forward is a stub): the
 * layouts of the upstream package's SSD interface, time-major:
 *   x, z, y : (batch, seqlen, nheads, headdim)    dt_raw : (batch, seqlen, nheads)
 *   B, C    : (batch, seqlen, ngroups, dstate)    A, D, dt_bias : (nheads)
 *   h0, h_last : (batch, nheads, headdim, dstate)
 * head h reads group h / (nheads / ngroups). z, D, dt_bias, h0, h_last may be NULL. */
int oracle_ssd_scan(const float *x, const float *dt_raw, const float *A, const float *B,
                    const float *C, const float *D, const float *z, const float *dt_bias,
                    int softplus, const double *h0, double *y, double *h_last, int64_t batch,
                    int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                    int64_t dstate, int nthreads) {
    if (batch < 0 || seqlen < 0 || nheads < 1 || headdim < 1 || ngroups < 1 || dstate < 1 ||
        nheads % ngroups != 0)
        return -1;
    int64_t H = nheads, P = headdim, G = ngroups, N = dstate, L = seqlen;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t bh = 0; bh < batch * H; bh++) {
        int64_t b = bh / H, h = bh % H, g = h / (H / G);
        double *S = (double *)malloc(sizeof(double) * (size_t)(P * N));
        for (int64_t k = 0; k < P * N; k++) S[k] = h0 ? h0[bh * P * N + k] : 0.0;
        for (int64_t t = 0; t < L; t++) {
            double v = (double)dt_raw[(b * L + t) * H + h] + (dt_bias ? (double)dt_bias[h] : 0.0);
            double dt = softplus ? oracle_softplus(v) : v;
            double a = exp(dt * (double)A[h]);
            const float *Bt = B + ((b * L + t) * G + g) * N, *Ct = C + ((b * L + t) * G + g) * N;
            for (int64_t p = 0; p < P; p++) {
                int64_t xi = ((b * L + t) * H + h) * P + p;
                double xt = (double)x[xi];
                double acc = 0.0;
                for (int64_t n = 0; n < N; n++) {
                    double *s = &S[p * N + n];
                    *s = a * *s + dt * (double)Bt[n] * xt;
                    acc += (double)Ct[n] * *s;
                }
                double yv = acc + (D ? (double)D[h] * xt : 0.0);
                if (z) yv *= oracle_silu((double)z[xi]);
                y[xi] = yv;
            }
        }
        if (h_last)
            for (int64_t k = 0; k < P * N; k++) h_last[bh * P * N + k] = S[k];
        free(S);
    }
    return 0;
}

/* Causal depthwise 1-D convolution and SiLU: the step before the scan in the
 * same page's MambaBlock (section 5, "complete Mamba implementation"): __init__
 * builds nn.Conv1d(d_inner, d_inner, kernel_size=d_conv, groups=d_inner,
 * padding=d_conv - 1, bias=True) and forward keeps the first seqlen outputs of
 * the convolution and applies silu. PyTorch's Conv1d is a cross-correlation over
 * the input padded with width-1 zeros on the left, so with xp the padded input
 * (xp[j] = x[j - (width-1)], zero for j < width-1):
 *     out[t] = bias[d] + sum_{k=0}^{width-1} w[d][k] * xp[t + k]
 * w[d][width-1] multiplies the current input x[t]. Reading for the state the
 * page leaves open (chunked prefill, decode): the zero padding is replaced by
 * the width-1 inputs that preceded this call, oldest first (conv_state_in;
 * zeros when NULL), and conv_state_out receives the last width-1 entries of the
 * padded input, i.e. the state a following call continues from.
 *   x, out : (batch, dim, seqlen)     w : (dim, width)     bias : (dim) or NULL
 *   conv_state_in, conv_state_out : (batch, dim, width - 1) or NULL
 */
int oracle_causal_conv1d(const float *x, const float *w, const float *bias,
                         const double *conv_state_in, int silu, double *out,
                         double *conv_state_out, int64_t batch, int64_t dim, int64_t seqlen,
                         int64_t width, int nthreads) {
    if (batch < 0 || dim < 0 || seqlen < 0 || width < 1) return -1;
    int64_t nch = batch * dim, hw = width - 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t ch = 0; ch < nch; ch++) {
        int64_t d = ch % dim;
        /* the padded input of this channel: width-1 state entries, then x */
        double *xp = (double *)malloc(sizeof(double) * (size_t)(hw + seqlen + 1));
        for (int64_t j = 0; j < hw; j++) xp[j] = conv_state_in ? conv_state_in[ch * hw + j] : 0.0;
        for (int64_t t = 0; t < seqlen; t++) xp[hw + t] = (double)x[ch * seqlen + t];
        for (int64_t t = 0; t < seqlen; t++) {
            double acc = bias ? (double)bias[d] : 0.0;
            for (int64_t k = 0; k < width; k++) acc += (double)w[d * width + k] * xp[t + k];
            out[ch * seqlen + t] = silu ? oracle_silu(acc) : acc;
        }
        if (conv_state_out)
            for (int64_t j = 0; j < hw; j++) conv_state_out[ch * hw + j] = xp[seqlen + j];
        free(xp);
    }
    return 0;
}

/* One decode token of the same convolution, in place on the state (the width-1
 * most recent inputs, oldest first): out = bias + sum_{k<width-1} w[k] state[k]
 * + w[width-1] x, optionally silu; then the state drops its oldest entry and
 * appends x.
 *   conv_state : (batch, dim, width - 1) in/out   x, out : (batch, dim)
 */
int oracle_conv_update(double *conv_state, const float *x, const float *w, const float *bias,
                       int silu, double *out, int64_t batch, int64_t dim, int64_t width,
                       int nthreads) {
    if (batch < 0 || dim < 0 || width < 1) return -1;
    int64_t nch = batch * dim, hw = width - 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t ch = 0; ch < nch; ch++) {
        int64_t d = ch % dim;
        double *s = conv_state + ch * hw;
        double xt = (double)x[ch];
        double acc = bias ? (double)bias[d] : 0.0;
        for (int64_t k = 0; k < hw; k++) acc += (double)w[d * width + k] * s[k];
        acc += (double)w[d * width + hw] * xt;
        out[ch] = silu ? oracle_silu(acc) : acc;
        for (int64_t k = 0; k + 1 < hw; k++) s[k] = s[k + 1];
        if (hw > 0) s[hw - 1] = xt;
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
