/*
 * mamba3_oracle.c -- fp64 CPU oracle of the complex-valued selective scan
 * (the Mamba-3 state update).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA path is checked against.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark may load it; the
 * library itself never does.  It shares no code, header or constant with the
 * CUDA sources.
 *
 * Source: the lesson "Jamba -- SSM-Transformer Hibrido"
 * (ai-engineering.academy), section "Mamba-3: a linha de base de SSM puro em
 * 2026", items 1 and 2, which print no formula.  The reading taken here:
 *
 *  - Item 2 (complex-valued state update): the Mamba layer of
 *    "【大模型】- Jamba 混合 SSM-Transformer", section "实现 > Mamba 层"
 *    (conv1d -> silu -> softplus(dt) -> scan -> D skip -> silu(z) gate), with
 *    its diagonal state made complex: M complex modes per channel (2M reals,
 *    the state size of the real scan with d_state = 2M), each with
 *    lambda_n = -exp(A_log[c,n]) + i*theta[c,n].  The step's factor
 *    exp(dt*lambda_n) decays the mode and turns it by the data-dependent angle
 *    dt*theta_n -- the data-dependent rotation of the state the item names.
 *    B and C rows hold M complex numbers each as (re, im) pairs; the
 *    read-out is the real part of sum_n C_n h_n.
 *  - Item 1 (exponential-trapezoidal discretization): the state input
 *    v_t = B_t u_t enters through the trapezoidal rule over the step instead
 *    of Euler's right end point, the step's exact decay applied to the earlier
 *    end: h_t = alpha_t (h_{t-1} + dt_t/2 v_{t-1}) + dt_t/2 v_t -- a two-tap
 *    combination of consecutive state inputs inside the recurrence (the
 *    "convolution-like operation on the state input" of the item).  Euler
 *    (h_t = alpha_t h_{t-1} + dt_t v_t) stays available; v before the first
 *    token comes from v0 (or is zero).
 *
 * Per batch row b and channel c, for t = 0 .. L-1 (s: the K-1 previous
 * inputs, oldest first):
 *   pre   = conv_b + sum_k w[k] s_k + w[K-1] x_t;   u = silu(pre)
 *   dt    = softplus(dt_raw)                     (beta 1, threshold 20)
 *   alpha = exp(dt * lambda_n)                   (complex)
 *   v_n   = (B_re + i B_im)[t,n] * u
 *   h_n   = alpha h_n + dt v_n                              (Euler)
 *         | alpha (h_n + dt/2 vprev_n) + dt/2 v_n           (trapezoidal)
 *   y_t   = (Re(sum_n (C_re + i C_im)[t,n] h_n) + D u) * silu(z_t)
 *   vprev = v;  s = (s_1, .., x_t)
 *
 * Layouts (row-major, fp64, contiguous): x, z, dt_raw, y (B,L,D); Bm, Cm
 * (B,L,2M); A_log, theta (D,M); Dskip, conv_b (D); conv_w (D,K); h0,
 * final_h, v0, final_v (B,D,2M) as (re, im) pairs; conv_state0,
 * final_conv_state (B,K-1,D).  conv_b, h0, v0, conv_state0 may be NULL
 * (zeros); the final_* outputs may be NULL (not written).
 */
#include <complex.h>
#include <math.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double silu3(double v) { return v / (1.0 + exp(-v)); }

static double softplus3(double v) { return v > 20.0 ? v : log1p(exp(v)); }

/*
 * The complex recurrence of one row given its inputs u and dt directly (no
 * conv, softplus or gate): h (M complex) and vprev (M complex) are updated in
 * place; returns Re(sum_n C_n h_n) after the token.  trap: 0 Euler,
 * 1 trapezoidal.
 */
static double m3_step(int M, double complex *h, double complex *vprev, double u, double dt,
                      const double *Bt, const double *Ct, const double *A_log_c,
                      const double *theta_c, int trap)
{
    double ys = 0.0;
    for (int n = 0; n < M; ++n) {
        double complex lam = -exp(A_log_c[n]) + I * theta_c[n];
        double complex alpha = cexp(dt * lam);
        double complex v = (Bt[2 * n] + I * Bt[2 * n + 1]) * u;
        if (trap)
            h[n] = alpha * (h[n] + 0.5 * dt * vprev[n]) + 0.5 * dt * v;
        else
            h[n] = alpha * h[n] + dt * v;
        vprev[n] = v;
        ys += creal((Ct[2 * n] + I * Ct[2 * n + 1]) * h[n]);
    }
    return ys;
}

/*
 * The bare recurrence over L tokens of one row (test hook for the pins that
 * drive it with chosen u and dt): u, dt (L); Bm, Cm (L, 2M); h and v (2M
 * reals, in: initial state and previous input, out: final ones); ys (L).
 */
void oracle_m3_core_f64(int L, int M, const double *u, const double *dt,
                        const double *Bm, const double *Cm,
                        const double *A_log, const double *theta, int trap,
                        double *h, double *v, double *ys)
{
    double complex *hc = (double complex *)calloc((size_t)M, sizeof(double complex));
    double complex *vc = (double complex *)calloc((size_t)M, sizeof(double complex));
    for (int n = 0; n < M; ++n) {
        hc[n] = h[2 * n] + I * h[2 * n + 1];
        vc[n] = v[2 * n] + I * v[2 * n + 1];
    }
    for (int t = 0; t < L; ++t)
        ys[t] = m3_step(M, hc, vc, u[t], dt[t], Bm + (size_t)t * 2 * M, Cm + (size_t)t * 2 * M,
                        A_log, theta, trap);
    for (int n = 0; n < M; ++n) {
        h[2 * n] = creal(hc[n]);
        h[2 * n + 1] = cimag(hc[n]);
        v[2 * n] = creal(vc[n]);
        v[2 * n + 1] = cimag(vc[n]);
    }
    free(hc);
    free(vc);
}

static void m3_row(int b, int c, int L, int D, int M, int K, const double *x, const double *z,
                   const double *dt_raw, const double *Bm, const double *Cm, const double *A_log,
                   const double *theta, const double *Dskip, const double *conv_w,
                   const double *conv_b, const double *h0, const double *conv_state0,
                   const double *v0, int trap, double *y, double *final_h,
                   double *final_conv_state, double *final_v)
{
    double complex *h = (double complex *)calloc((size_t)M, sizeof(double complex));
    double complex *vp = (double complex *)calloc((size_t)M, sizeof(double complex));
    double *s = (double *)calloc((size_t)(K > 1 ? K - 1 : 1), sizeof(double));
    const size_t hs = ((size_t)b * D + c) * 2 * M;
    for (int n = 0; n < M; ++n) {
        if (h0) h[n] = h0[hs + 2 * n] + I * h0[hs + 2 * n + 1];
        if (v0) vp[n] = v0[hs + 2 * n] + I * v0[hs + 2 * n + 1];
    }
    if (conv_state0)
        for (int k = 0; k < K - 1; ++k) s[k] = conv_state0[((size_t)b * (K - 1) + k) * D + c];
    const double bias = conv_b ? conv_b[c] : 0.0;
    const double *w = conv_w + (size_t)c * K;

    for (int t = 0; t < L; ++t) {
        const size_t e = ((size_t)b * L + t) * D + c;
        const size_t r = ((size_t)b * L + t) * 2 * M;
        double pre = bias;
        for (int k = 0; k < K - 1; ++k) pre += w[k] * s[k];
        pre += w[K - 1] * x[e];
        const double u = silu3(pre);
        const double dt = softplus3(dt_raw[e]);
        const double ys = m3_step(M, h, vp, u, dt, Bm + r, Cm + r, A_log + (size_t)c * M,
                                  theta + (size_t)c * M, trap);
        y[e] = (ys + Dskip[c] * u) * silu3(z[e]);
        for (int k = 0; k + 1 < K - 1; ++k) s[k] = s[k + 1];
        if (K > 1) s[K - 2] = x[e];
    }
    for (int n = 0; n < M; ++n) {
        if (final_h) {
            final_h[hs + 2 * n] = creal(h[n]);
            final_h[hs + 2 * n + 1] = cimag(h[n]);
        }
        if (final_v) {
            final_v[hs + 2 * n] = creal(vp[n]);
            final_v[hs + 2 * n + 1] = cimag(vp[n]);
        }
    }
    if (final_conv_state)
        for (int k = 0; k < K - 1; ++k) final_conv_state[((size_t)b * (K - 1) + k) * D + c] = s[k];
    free(h);
    free(vp);
    free(s);
}

/* The complex scan over all (b, c) rows (independent; spread over threads). */
void oracle_m3_scan_f64(int batch, int seqlen, int d_inner, int modes, int d_conv,
                        const double *x, const double *z, const double *dt_raw,
                        const double *Bm, const double *Cm, const double *A_log,
                        const double *theta, const double *Dskip, const double *conv_w,
                        const double *conv_b, const double *h0, const double *conv_state0,
                        const double *v0, int trap, double *y, double *final_h,
                        double *final_conv_state, double *final_v, int n_threads)
{
    long rows = (long)batch * d_inner;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long i = 0; i < rows; ++i)
        m3_row((int)(i / d_inner), (int)(i % d_inner), seqlen, d_inner, modes, d_conv, x, z,
               dt_raw, Bm, Cm, A_log, theta, Dskip, conv_w, conv_b, h0, conv_state0, v0, trap,
               y, final_h, final_conv_state, final_v);
    (void)n_threads;
}
