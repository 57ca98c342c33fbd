/*
 * mamba_oracle.c -- fp64 CPU oracle of the Mamba selective-scan layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA path is checked against.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark may load it; the
 * library itself never does.  It shares no code, header or constant with the
 * CUDA sources.
 *
 * What it computes (per batch row b and channel c, sequential in t), from
 *   "【大模型】- Jamba 混合 SSM-Transformer" (sxl-space.tk), section
 *   "实现 > Mamba 层": MambaBlock.forward (conv1d -> silu -> dt_proj ->
 *   softplus -> ssm -> y * silu(z)) and MambaBlock.ssm (dA = exp(dt*A),
 *   dB = dt*B, h = dA*h + dB*x),
 * with the read-out taken from the lesson "Jamba -- SSM-Transformer Hibrido"
 *   (ai-engineering.academy / aiengineeringfromscratch.com), section
 *   "Um SSM em uma pagina": y_t = C h_t.  The blog's `(h*D).sum(-1)`
 *   read-out is a slip; the definition used here is y_t = C_t.h_t + D*u_t.
 *
 *   pre  = conv_b + w[0]*s0 + w[1]*s1 + w[2]*s2 + w[K-1]*x_t
 *          (causal depthwise cross-correlation: PyTorch Conv1d with
 *           padding K-1 truncated to the first L outputs; s = the K-1
 *           previous inputs, zeros before the sequence start)
 *   u    = silu(pre) = pre / (1 + exp(-pre))
 *   dt   = softplus(dt_raw) = dt_raw > 20 ? dt_raw : log1p(exp(dt_raw))
 *          (F.softplus defaults: beta = 1, threshold = 20)
 *   A_n  = -exp(A_log[c,n])
 *   h_n  = exp(dt*A_n) * h_n + (dt*B[t,n]) * u      n = 0..N-1
 *   y_t  = (sum_n C[t,n]*h_n + D[c]*u) * silu(z_t)
 *   s    = (s1, ..., s_{K-2}, x_t)
 *
 * Outputs: y (B,L,D); final_h (B,D,N) = h after the last token;
 * final_conv_state (B,K-1,D) = s after the last token (the last K-1 inputs,
 * earlier ones taken from conv_state0 when L < K-1).
 *
 * Layouts (all row-major, fp64, contiguous):
 *   x, z, dt_raw, y      (B, L, D)
 *   Bm, Cm               (B, L, N)
 *   A_log                (D, N)
 *   Dskip, conv_b        (D)
 *   conv_w               (D, K)
 *   h0, final_h          (B, D, N)
 *   conv_state0, final_conv_state  (B, K-1, D)
 * conv_b, h0 and conv_state0 may be NULL (read as zeros).  final_h and
 * final_conv_state may be NULL (not written).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double silu(double v) { return v / (1.0 + exp(-v)); }

static double softplus(double v) { return v > 20.0 ? v : log1p(exp(v)); }

/*
 * One token of one (b, c) row: the loop body of the scan.  h has N entries;
 * s holds the K-1 previous inputs, oldest first.  Returns y_t.
 */
static double token_update(int N, int K, double *h, double *s,
                           double x, double z, double dt_raw,
                           const double *Bt, const double *Ct,
                           const double *A_log_c, double Dc,
                           const double *w_c, double bias)
{
    /* causal depthwise conv: w[k] multiplies the input k-(K-1) steps back */
    double pre = bias;
    for (int k = 0; k < K - 1; ++k) pre += w_c[k] * s[k];
    pre += w_c[K - 1] * x;
    double u = silu(pre);

    double dt = softplus(dt_raw);
    double yss = 0.0;
    for (int n = 0; n < N; ++n) {
        double A = -exp(A_log_c[n]);
        double dA = exp(dt * A);
        double dB = dt * Bt[n];
        h[n] = dA * h[n] + dB * u;
        yss += Ct[n] * h[n];
    }
    yss += Dc * u;

    for (int k = 0; k + 1 < K - 1; ++k) s[k] = s[k + 1];
    if (K > 1) s[K - 2] = x;
    return yss * silu(z);
}

/* the (b, c) row of the scan, t = 0 .. L-1 */
static void scan_row(int b, int c, int L, int D, int N, int K,
                     const double *x, const double *z, const double *dt_raw,
                     const double *Bm, const double *Cm,
                     const double *A_log, const double *Dskip,
                     const double *conv_w, const double *conv_b,
                     const double *h0, const double *conv_state0,
                     double *y, double *final_h, double *final_conv_state)
{
    double *h = (double *)calloc((size_t)N, sizeof(double));
    double *s = (double *)calloc((size_t)(K > 1 ? K - 1 : 1), sizeof(double));
    if (h0)
        for (int n = 0; n < N; ++n) h[n] = h0[((size_t)b * D + c) * N + n];
    if (conv_state0)
        for (int k = 0; k < K - 1; ++k)
            s[k] = conv_state0[((size_t)b * (K - 1) + k) * D + c];
    double bias = conv_b ? conv_b[c] : 0.0;

    for (int t = 0; t < L; ++t) {
        size_t e = ((size_t)b * L + t) * D + c;
        size_t r = ((size_t)b * L + t) * N;
        y[e] = token_update(N, K, h, s, x[e], z[e], dt_raw[e], Bm + r, Cm + r,
                            A_log + (size_t)c * N, Dskip[c],
                            conv_w + (size_t)c * K, bias);
    }
    if (final_h)
        for (int n = 0; n < N; ++n) final_h[((size_t)b * D + c) * N + n] = h[n];
    if (final_conv_state)
        for (int k = 0; k < K - 1; ++k)
            final_conv_state[((size_t)b * (K - 1) + k) * D + c] = s[k];
    free(h);
    free(s);
}

/*
 * Sequential selective scan over all (b, c) rows.  Rows are independent, so
 * they are spread over n_threads OpenMP threads (n_threads <= 0: the OpenMP
 * default); each row is still the plain sequential loop above.
 */
void oracle_scan_f64(int batch, int seqlen, int d_inner, int d_state, int d_conv,
                     const double *x, const double *z, const double *dt_raw,
                     const double *Bm, const double *Cm,
                     const double *A_log, const double *Dskip,
                     const double *conv_w, const double *conv_b,
                     const double *h0, const double *conv_state0,
                     double *y, double *final_h, double *final_conv_state,
                     int n_threads)
{
    long rows = (long)batch * d_inner;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long i = 0; i < rows; ++i) {
        int b = (int)(i / d_inner), c = (int)(i % d_inner);
        scan_row(b, c, seqlen, d_inner, d_state, d_conv, x, z, dt_raw, Bm, Cm,
                 A_log, Dskip, conv_w, conv_b, h0, conv_state0, y, final_h,
                 final_conv_state);
    }
    (void)n_threads;
}

/*
 * One decode token for every (b, c): the same loop body as the scan, applied
 * in place to h (B,D,N) and conv_state (B,K-1,D).  x_t, z_t, dt_raw_t and y_t
 * are (B,D); B_t and C_t are (B,N).  The lesson's "Um SSM em uma pagina":
 * y_t needs only h_{t-1} and x_t, O(1) memory per token.
 */
void oracle_step_f64(int batch, int d_inner, int d_state, int d_conv,
                     double *h, double *conv_state,
                     const double *x_t, const double *z_t, const double *dt_raw_t,
                     const double *B_t, const double *C_t,
                     const double *A_log, const double *Dskip,
                     const double *conv_w, const double *conv_b,
                     double *y_t)
{
    int D = d_inner, N = d_state, K = d_conv;
    double *s = (double *)calloc((size_t)(K > 1 ? K - 1 : 1), sizeof(double));
    for (int b = 0; b < batch; ++b)
        for (int c = 0; c < D; ++c) {
            for (int k = 0; k < K - 1; ++k)
                s[k] = conv_state[((size_t)b * (K - 1) + k) * D + c];
            size_t e = (size_t)b * D + c;
            y_t[e] = token_update(N, K, h + e * N, s, x_t[e], z_t[e], dt_raw_t[e],
                                  B_t + (size_t)b * N, C_t + (size_t)b * N,
                                  A_log + (size_t)c * N, Dskip[c],
                                  conv_w + (size_t)c * K, conv_b ? conv_b[c] : 0.0);
            for (int k = 0; k < K - 1; ++k)
                conv_state[((size_t)b * (K - 1) + k) * D + c] = s[k];
        }
    free(s);
}

/* input of row (b, c) at time tau, taken from conv_state0 (or 0) for tau < 0 */
static double input_at(int b, int c, long tau, int L, int D, int K,
                       const double *x, const double *conv_state0)
{
    if (tau >= 0) return x[((size_t)b * L + (size_t)tau) * D + c];
    long k = tau + (K - 1);
    if (!conv_state0 || k < 0) return 0.0;
    return conv_state0[((size_t)b * (K - 1) + (size_t)k) * D + c];
}

/*
 * The same scan evaluated chunk by chunk, as a check that splitting the
 * sequence and carrying the decayed chunk state gives the sequential result.
 * With chunks of `chunk` tokens, for chunk j and state n:
 *   P_j[n]    = exp(A_n * sum_{t in chunk j} dt_t)   decay across the chunk
 *   hloc_j[n] = end state of chunk j started from h = 0
 *   H_j       = P_j[n] * H_{j-1}[n] + hloc_j[n],  H_{-1} = h0
 * (a fixed left fold in chunk order), and y inside chunk j is recomputed
 * starting from h = H_{j-1}.  final_h is the fold value H_last.
 */
void oracle_scan_chunked_f64(int batch, int seqlen, int d_inner, int d_state, int d_conv,
                             int chunk,
                             const double *x, const double *z, const double *dt_raw,
                             const double *Bm, const double *Cm,
                             const double *A_log, const double *Dskip,
                             const double *conv_w, const double *conv_b,
                             const double *h0, const double *conv_state0,
                             double *y, double *final_h, double *final_conv_state)
{
    int L = seqlen, D = d_inner, N = d_state, K = d_conv;
    int n_chunks = (L + chunk - 1) / chunk;
    double *H = (double *)calloc((size_t)(n_chunks + 1) * N, sizeof(double));
    double *h = (double *)calloc((size_t)N, sizeof(double));
    double *s = (double *)calloc((size_t)(K > 1 ? K - 1 : 1), sizeof(double));
    double *P = (double *)calloc((size_t)N, sizeof(double));
    for (int b = 0; b < batch; ++b)
        for (int c = 0; c < D; ++c) {
            const double *Al = A_log + (size_t)c * N;
            const double *w = conv_w + (size_t)c * K;
            double bias = conv_b ? conv_b[c] : 0.0;
            /* H[0] is the carry into chunk 0 (h0), H[j+1] the carry out of chunk j */
            for (int n = 0; n < N; ++n)
                H[n] = h0 ? h0[((size_t)b * D + c) * N + n] : 0.0;
            for (int j = 0; j < n_chunks; ++j) {
                int t0 = j * chunk, t1 = t0 + chunk < L ? t0 + chunk : L;
                for (int n = 0; n < N; ++n) h[n] = 0.0;
                for (int k = 0; k < K - 1; ++k)
                    s[k] = input_at(b, c, (long)t0 - (K - 1) + k, L, D, K, x, conv_state0);
                double sum_dt = 0.0;
                for (int t = t0; t < t1; ++t) {
                    size_t e = ((size_t)b * L + t) * D + c, r = ((size_t)b * L + t) * N;
                    (void)token_update(N, K, h, s, x[e], z[e], dt_raw[e], Bm + r, Cm + r,
                                       Al, Dskip[c], w, bias);
                    sum_dt += softplus(dt_raw[e]);
                }
                for (int n = 0; n < N; ++n) {
                    P[n] = exp(-exp(Al[n]) * sum_dt);
                    H[(size_t)(j + 1) * N + n] = P[n] * H[(size_t)j * N + n] + h[n];
                }
            }
            for (int j = 0; j < n_chunks; ++j) {
                int t0 = j * chunk, t1 = t0 + chunk < L ? t0 + chunk : L;
                for (int n = 0; n < N; ++n) h[n] = H[(size_t)j * N + n];
                for (int k = 0; k < K - 1; ++k)
                    s[k] = input_at(b, c, (long)t0 - (K - 1) + k, L, D, K, x, conv_state0);
                for (int t = t0; t < t1; ++t) {
                    size_t e = ((size_t)b * L + t) * D + c, r = ((size_t)b * L + t) * N;
                    y[e] = token_update(N, K, h, s, x[e], z[e], dt_raw[e], Bm + r, Cm + r,
                                        Al, Dskip[c], w, bias);
                }
            }
            if (final_h)
                for (int n = 0; n < N; ++n)
                    final_h[((size_t)b * D + c) * N + n] = H[(size_t)n_chunks * N + n];
            if (final_conv_state)
                for (int k = 0; k < K - 1; ++k)
                    final_conv_state[((size_t)b * (K - 1) + k) * D + c] =
                        input_at(b, c, (long)L - (K - 1) + k, L, D, K, x, conv_state0);
        }
    free(H); free(h); free(s); free(P);
}

/* ------------------------------------------------------------------ backward
 *
 * Reverse-mode gradient of the scan above (the next step for training; the
 * pages train the layer end to end, "【大模型】- Jamba 混合 SSM-Transformer",
 * section "训练" / Jamba.forward's cross-entropy loss, but print no backward:
 * this is the chain rule applied to the forward definition, written out).
 * For the scalar
 *   loss = sum y*dy + sum final_h*dfinal_h + sum final_conv_state*dfinal_conv_state
 * it returns the gradients with respect to every input.  Per (b, c) row the
 * forward pass is run first, keeping every state; then t runs backwards with
 * lam = d loss / d h_t:
 *   dyss = dy*silu(z);   dz = dy*yss*silu'(z)
 *   lam += C_t*dyss;     dC_t += dyss*h_t;     du = dyss*D;   dD += dyss*u
 *   for each n:  g = lam*h_{t-1};  ddt += g*dA*A + lam*B*u;
 *                dA_log += g*dA*dt*A   (A = -exp(A_log), dA = exp(dt*A));
 *                dB_t += lam*dt*u;  du += lam*dt*B;  lam *= dA
 *   ddt_raw = ddt * softplus'(dt_raw)    (sigmoid, or 1 above the threshold)
 *   dpre = du*silu'(pre);  dconv_b += dpre;  dconv_w[k] += dpre*in(t-K+1+k);
 *   d in(t-K+1+k) += dpre*w[k]
 * and at the end dh0 = lam; inputs before t = 0 send their gradient to
 * dconv_state0.  silu'(v) = s(1 + v(1 - s)), s = sigmoid(v).
 *
 * All gradient outputs are overwritten (zeroed first).  dfinal_h and
 * dfinal_conv_state may be NULL (zero).  Single-threaded: the B and C
 * gradients sum over channels.
 */
static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

static double dsilu(double v)
{
    double s = sigmoid(v);
    return s * (1.0 + v * (1.0 - s));
}

static double dsoftplus(double v) { return v > 20.0 ? 1.0 : sigmoid(v); }

void oracle_scan_bwd_f64(int batch, int seqlen, int d_inner, int d_state, int d_conv,
                         const double *x, const double *z, const double *dt_raw,
                         const double *Bm, const double *Cm,
                         const double *A_log, const double *Dskip,
                         const double *conv_w, const double *conv_b,
                         const double *h0, const double *conv_state0,
                         const double *dy, const double *dfinal_h,
                         const double *dfinal_conv_state,
                         double *dx, double *dz, double *ddt_raw,
                         double *dB, double *dC, double *dA_log, double *dD,
                         double *dconv_w, double *dconv_b, double *dh0,
                         double *dconv_state0)
{
    int L = seqlen, D = d_inner, N = d_state, K = d_conv, B = batch;
    size_t nLD = (size_t)B * L * D, nLN = (size_t)B * L * N;
    memset(dx, 0, nLD * sizeof(double));
    memset(dz, 0, nLD * sizeof(double));
    memset(ddt_raw, 0, nLD * sizeof(double));
    memset(dB, 0, nLN * sizeof(double));
    memset(dC, 0, nLN * sizeof(double));
    memset(dA_log, 0, (size_t)D * N * sizeof(double));
    memset(dD, 0, (size_t)D * sizeof(double));
    memset(dconv_w, 0, (size_t)D * K * sizeof(double));
    memset(dconv_b, 0, (size_t)D * sizeof(double));
    memset(dh0, 0, (size_t)B * D * N * sizeof(double));
    if (K > 1) memset(dconv_state0, 0, (size_t)B * (K - 1) * D * sizeof(double));

    double *hs = (double *)malloc((size_t)(L + 1) * N * sizeof(double)); /* hs[t+1] = h after t */
    double *u = (double *)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    double *pre = (double *)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    double *dt = (double *)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    double *yss = (double *)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    double *din = (double *)malloc((size_t)(L + K) * sizeof(double)); /* d in(tau), tau = -(K-1) .. L-1 */
    double *lam = (double *)malloc((size_t)N * sizeof(double));

    for (int b = 0; b < B; ++b)
        for (int c = 0; c < D; ++c) {
            const double *Al = A_log + (size_t)c * N;
            const double *w = conv_w + (size_t)c * K;
            double bias = conv_b ? conv_b[c] : 0.0;
            /* forward, keeping every state */
            for (int n = 0; n < N; ++n) hs[n] = h0 ? h0[((size_t)b * D + c) * N + n] : 0.0;
            for (int t = 0; t < L; ++t) {
                size_t e = ((size_t)b * L + t) * D + c, r = ((size_t)b * L + t) * N;
                double p = bias;
                for (int k = 0; k < K; ++k)
                    p += w[k] * input_at(b, c, (long)t - (K - 1) + k, L, D, K, x, conv_state0);
                pre[t] = p;
                u[t] = silu(p);
                dt[t] = softplus(dt_raw[e]);
                double acc = 0.0;
                for (int n = 0; n < N; ++n) {
                    double A = -exp(Al[n]);
                    double hn = exp(dt[t] * A) * hs[(size_t)t * N + n] + dt[t] * Bm[r + n] * u[t];
                    hs[(size_t)(t + 1) * N + n] = hn;
                    acc += Cm[r + n] * hn;
                }
                yss[t] = acc + Dskip[c] * u[t];
            }
            /* backward */
            for (int i = 0; i < L + K; ++i) din[i] = 0.0;
            if (dfinal_conv_state)
                for (int k = 0; k < K - 1; ++k)
                    din[(L - (K - 1) + k) + (K - 1)] +=
                        dfinal_conv_state[((size_t)b * (K - 1) + k) * D + c];
            for (int n = 0; n < N; ++n)
                lam[n] = dfinal_h ? dfinal_h[((size_t)b * D + c) * N + n] : 0.0;
            for (int t = L - 1; t >= 0; --t) {
                size_t e = ((size_t)b * L + t) * D + c, r = ((size_t)b * L + t) * N;
                double g = silu(z[e]);
                double dyss = dy[e] * g;
                dz[e] = dy[e] * yss[t] * dsilu(z[e]);
                double du = dyss * Dskip[c];
                dD[c] += dyss * u[t];
                double ddt = 0.0;
                for (int n = 0; n < N; ++n) {
                    lam[n] += Cm[r + n] * dyss;
                    dC[r + n] += dyss * hs[(size_t)(t + 1) * N + n];
                    double A = -exp(Al[n]);
                    double dA = exp(dt[t] * A);
                    double gA = lam[n] * hs[(size_t)t * N + n];
                    ddt += gA * dA * A + lam[n] * Bm[r + n] * u[t];
                    dA_log[(size_t)c * N + n] += gA * dA * dt[t] * A;
                    dB[r + n] += lam[n] * dt[t] * u[t];
                    du += lam[n] * dt[t] * Bm[r + n];
                    lam[n] *= dA;
                }
                ddt_raw[e] = ddt * dsoftplus(dt_raw[e]);
                double dpre = du * dsilu(pre[t]);
                if (conv_b) dconv_b[c] += dpre;
                for (int k = 0; k < K; ++k) {
                    long tau = (long)t - (K - 1) + k;
                    dconv_w[(size_t)c * K + k] +=
                        dpre * input_at(b, c, tau, L, D, K, x, conv_state0);
                    din[tau + (K - 1)] += dpre * w[k];
                }
            }
            for (int n = 0; n < N; ++n) dh0[((size_t)b * D + c) * N + n] = lam[n];
            for (long tau = -(K - 1); tau < L; ++tau) {
                double v = din[tau + (K - 1)];
                if (tau >= 0)
                    dx[((size_t)b * L + (size_t)tau) * D + c] = v;
                else
                    dconv_state0[((size_t)b * (K - 1) + (size_t)(tau + (K - 1))) * D + c] = v;
            }
        }
    free(hs); free(u); free(pre); free(dt); free(yss); free(din); free(lam);
}

/*
 * Mamba-2's structure ("Jamba -- SSM-Transformer Hibrido", ai-engineering.academy,
 * section "Mamba-3: a linha de base de SSM puro em 2026", items 1 and 2: Mamba-2
 * reduced the state matrix to a scaled identity and discretises with Euler's
 * method): the channels come in heads of P that share one scalar decay
 * exp(dt*A_h) per token, dt and A being per head, and one state matrix of
 * N x P per head.  For batch row b, head h (group g = h / (H / G) of the B and
 * C rows), t = 0..L-1:
 *   dt       = softplus(dt_raw[b,t,h])            (beta 1, threshold 20)
 *   S[n][p]  = exp(dt * A_h) * S[n][p] + dt * B[b,t,g,n] * x[b,t,h,p]
 *   y[p]     = (sum_n C[b,t,g,n] * S[n][p] + D_h * x[b,t,h,p]) * silu(z[b,t,h,p])
 * with A_h = -exp(A_log[h]), S starting at h0[b,h] (or zero), the gate only
 * when z is given.  Layouts: x, z, y (B,L,H,P); dt_raw (B,L,H); Bm, Cm
 * (B,L,G,N); A_log, Dskip (H); h0, final_S (B,H,N,P).  Plain sequential fp64.
 */
void oracle_ssd_f64(int batch, int seqlen, int heads, int head_dim, int groups, int d_state,
                    const double *x, const double *z, const double *dt_raw, const double *A_log,
                    const double *Bm, const double *Cm, const double *Dskip, const double *h0,
                    double *y, double *final_S)
{
    int B = batch, L = seqlen, H = heads, P = head_dim, G = groups, N = d_state;
    int hpg = H / G;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            int g = h / hpg;
            double *S = (double *)malloc((size_t)N * P * sizeof(double));
            for (int i = 0; i < N * P; ++i)
                S[i] = h0 ? h0[((size_t)b * H + h) * N * P + i] : 0.0;
            double A = -exp(A_log[h]);
            for (int t = 0; t < L; ++t) {
                double dt = softplus(dt_raw[((size_t)b * L + t) * H + h]);
                double a = exp(dt * A);
                const double *xr = x + (((size_t)b * L + t) * H + h) * P;
                const double *Br = Bm + (((size_t)b * L + t) * G + g) * N;
                const double *Cr = Cm + (((size_t)b * L + t) * G + g) * N;
                for (int n = 0; n < N; ++n)
                    for (int p = 0; p < P; ++p)
                        S[n * P + p] = a * S[n * P + p] + dt * Br[n] * xr[p];
                for (int p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int n = 0; n < N; ++n) acc += Cr[n] * S[n * P + p];
                    double v = acc + Dskip[h] * xr[p];
                    if (z) v *= silu(z[(((size_t)b * L + t) * H + h) * P + p]);
                    y[(((size_t)b * L + t) * H + h) * P + p] = v;
                }
            }
            if (final_S)
                for (int i = 0; i < N * P; ++i) final_S[((size_t)b * H + h) * N * P + i] = S[i];
            free(S);
        }
}
