/*
 * ne_attn_oracle.c -- plain, slow CPU oracle for causal self-attention with
 * rotary position embedding (RoPE), forward and backward, in double precision;
 * also for the projections around it and for a multi-token prediction head
 * with its loss and gradients (each at the end of this file).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * path.  It is written for a reader checking it against the definitions:
 * every output element is computed straight from its formula, with no tiling,
 * no online softmax and no fusion.
 *
 * What it computes (per sequence of length L and per head, positions m,n in
 * 0..L-1; the pages print no equations, so the standard definitions are used):
 *
 *   RoPE (RoFormer, Su et al. 2021, in the rotate-half arrangement): for
 *   i < D/2, theta_i = base^(-(2i)/D), angle a = m * theta_i,
 *       x'_i       = x_i c - x_{i+D/2} s
 *       x'_{i+D/2} = x_{i+D/2} c + x_i s          (c = cos a, s = sin a)
 *   "Tiny Hackable CUDA" page, section 3: projections are computed, then RoPE
 *   encodes relative position; NanoEuler Show HN page, paragraph 2: the CUDA
 *   engine has RoPE beside a hand-written FlashAttention.
 *
 *   Causal scaled dot-product attention ("Tiny Hackable CUDA", section 3:
 *   each prediction depends only on earlier positions):
 *       S_mn   = scale * q'_m . k'_n                 for n <= m
 *       LSE_m  = log sum_{n<=m} exp(S_mn)            (natural log)
 *       P_mn   = exp(S_mn - LSE_m), and 0 for n > m
 *       O_m    = sum_n P_mn v_n
 *
 *   Analytic gradients (NanoEuler Show HN page, paragraph 2: every analytic
 *   gradient, including through RoPE, is checked against a double-precision
 *   centred finite difference; the tests here do the same to this file):
 *       dv_n   = sum_{m>=n} P_mn dO_m
 *       dP_mn  = dO_m . v_n
 *       D_m    = sum_n P_mn dP_mn
 *       dS_mn  = P_mn (dP_mn - D_m)
 *       dq_m   = R(m)^T ( scale * sum_n dS_mn k'_n )
 *       dk_n   = R(n)^T ( scale * sum_m dS_mn q'_m )
 *
 * Operand mode.  mode 0 keeps every quantity in double.  mode 1 models the
 * operands a bf16 tensor core consumes: the rotation is evaluated with fp32
 * cos/sin values (each the fp32 rounding of the double cos/sin above) as
 *       lo = fmaf(x_i, c, -(x_{i+D/2} * s)),   hi = fmaf(x_{i+D/2}, c, x_i * s)
 * in fp32, and the results are rounded to bf16 (round to nearest, ties to
 * even).  Everything after the rotation stays in double.  This is the only
 * place where the oracle follows the precision of the device: the bf16 code
 * of each rotated element is a rounding decision, and both sides take it in
 * the same precision.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (fp-contract off
 * keeps the fp32 products of mode 1 unfused).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Round a double to the nearest bf16 value (8 significant bits), ties to
 * even, directly (no intermediate float).  Inputs here are far from the bf16
 * subnormal and overflow ranges, which this does not model. */
static double round_to_bf16(double x)
{
    if (x == 0.0 || !isfinite(x))
        return x;
    int e;
    double f = frexp(x, &e);                 /* x = f * 2^e, 0.5 <= |f| < 1 */
    double r = nearbyint(ldexp(f, 8));       /* default mode: nearest, ties to even */
    return ldexp(r, e - 8);
}

/* Rotate one D-vector x (element stride 1) at position m. */
static void rope_vector(const double *x, int D, int m, double base, int mode, double *out)
{
    int half = D / 2;
    for (int i = 0; i < half; i++) {
        double theta = pow(base, -(2.0 * i) / D);
        double a = (double)m * theta;
        double c = cos(a), s = sin(a);
        double x0 = x[i], x1 = x[i + half];
        if (mode == 0) {
            out[i] = x0 * c - x1 * s;
            out[i + half] = x1 * c + x0 * s;
        } else {
            float cf = (float)c, sf = (float)s;
            float a0 = (float)x0, a1 = (float)x1;
            float p1 = a1 * sf;
            float p0 = a0 * sf;
            float lo = fmaf(a0, cf, -p1);
            float hi = fmaf(a1, cf, p0);
            out[i] = round_to_bf16((double)lo);
            out[i + half] = round_to_bf16((double)hi);
        }
    }
}

/* Apply R(m)^T to a gradient vector g' (always in double). */
static void rope_vector_transpose(const double *g, int D, int m, double base, double *out)
{
    int half = D / 2;
    for (int i = 0; i < half; i++) {
        double theta = pow(base, -(2.0 * i) / D);
        double a = (double)m * theta;
        double c = cos(a), s = sin(a);
        double g0 = g[i], g1 = g[i + half];
        out[i] = g0 * c + g1 * s;
        out[i + half] = -g0 * s + g1 * c;
    }
}

static double dot(const double *a, const double *b, int D)
{
    double acc = 0.0;
    for (int d = 0; d < D; d++)
        acc += a[d] * b[d];
    return acc;
}

/* Exported: rotate L rows (row stride `stride` elements) at positions 0..L-1
 * into out[L][D].  Returns 0, or -1 on bad arguments. */
int ne_oracle_rope(const double *x, long long stride, int L, int D, double base, int mode,
                   double *out)
{
    if (!x || !out || L < 0 || D <= 0 || (D % 2) != 0)
        return -1;
    for (int m = 0; m < L; m++)
        rope_vector(x + (long long)m * stride, D, m, base, mode, out + (long long)m * D);
    return 0;
}

/* Exported: apply R(m)^T at positions 0..L-1 (used by the tests' pins). */
int ne_oracle_rope_transpose(const double *g, long long stride, int L, int D, double base,
                             double *out)
{
    if (!g || !out || L < 0 || D <= 0 || (D % 2) != 0)
        return -1;
    for (int m = 0; m < L; m++)
        rope_vector_transpose(g + (long long)m * stride, D, m, base, out + (long long)m * D);
    return 0;
}

/* Row statistics of one query row m: LSE_m, and (when dout is given)
 * D_m = sum_n P_mn dP_mn.  s_buf holds L doubles. */
static void row_stats(const double *qr, const double *kr, const double *v, const double *dout,
                      long long stride, int D, double scale, int m, double *s_buf,
                      double *lse_out, double *delta_out, double *o_out)
{
    const double *qm = qr + (long long)m * D;
    double mx = -INFINITY;
    for (int n = 0; n <= m; n++) {
        s_buf[n] = scale * dot(qm, kr + (long long)n * D, D);
        if (s_buf[n] > mx)
            mx = s_buf[n];
    }
    double l = 0.0;
    for (int n = 0; n <= m; n++)
        l += exp(s_buf[n] - mx);
    double lse = mx + log(l);
    *lse_out = lse;
    if (o_out) {
        for (int d = 0; d < D; d++)
            o_out[d] = 0.0;
        for (int n = 0; n <= m; n++) {
            double p = exp(s_buf[n] - lse);
            const double *vn = v + (long long)n * stride;
            for (int d = 0; d < D; d++)
                o_out[d] += p * vn[d];
        }
    }
    if (delta_out) {
        const double *dom = dout + (long long)m * stride;
        double acc = 0.0;
        for (int n = 0; n <= m; n++) {
            double p = exp(s_buf[n] - lse);
            double dp = dot(dom, v + (long long)n * stride, D);
            acc += p * dp;
        }
        *delta_out = acc;
    }
}

/*
 * Exported: attention of one (sequence, head).
 *
 * q, k, v, dout point at row 0 of this sequence and head inside a
 * [tokens, heads, D] array; consecutive rows are `stride` doubles apart.
 * dout may be NULL (forward only).  qrows[nq] are the query rows whose
 * O (o[nq][D]), LSE (lse[nq]), D_m (delta[nq]) and dq (dq[nq][D]) are wanted;
 * krows[nk] are the key rows whose dk, dv (dk[nk][D], dv[nk][D]) are wanted.
 * Any output pointer may be NULL.  Returns 0, or -1 on bad arguments / OOM.
 */
int ne_oracle_attention_head(const double *q, const double *k, const double *v,
                             const double *dout, long long stride, int L, int D, double base,
                             double scale, int mode, const int *qrows, int nq, const int *krows,
                             int nk, double *o, double *lse, double *delta, double *dq,
                             double *dk, double *dv)
{
    if (!q || !k || !v || L <= 0 || D <= 0 || (D % 2) != 0 || nq < 0 || nk < 0)
        return -1;
    if ((nq > 0 && !qrows) || (nk > 0 && !krows))
        return -1;
    if (!dout && (dq || dk || dv || delta))
        return -1;
    for (int i = 0; i < nq; i++)
        if (qrows[i] < 0 || qrows[i] >= L)
            return -1;
    for (int i = 0; i < nk; i++)
        if (krows[i] < 0 || krows[i] >= L)
            return -1;

    double *qr = malloc(sizeof(double) * (size_t)L * D);
    double *kr = malloc(sizeof(double) * (size_t)L * D);
    double *lse_all = malloc(sizeof(double) * (size_t)L);
    double *delta_all = malloc(sizeof(double) * (size_t)L);
    char *need = calloc((size_t)L, 1);
    if (!qr || !kr || !lse_all || !delta_all || !need) {
        free(qr); free(kr); free(lse_all); free(delta_all); free(need);
        return -1;
    }
    ne_oracle_rope(q, stride, L, D, base, mode, qr);
    ne_oracle_rope(k, stride, L, D, base, mode, kr);

    /* Rows whose LSE_m / D_m are needed: the requested query rows, and for
     * key row n every query row m >= n. */
    int kmin = L;
    for (int i = 0; i < nk; i++)
        if (krows[i] < kmin)
            kmin = krows[i];
    for (int i = 0; i < nq; i++)
        need[qrows[i]] = 1;
    for (int m = kmin; m < L; m++)
        need[m] = 1;

    int failed = 0;
#pragma omp parallel
    {
        double *s_buf = malloc(sizeof(double) * (size_t)L);
        double *g = malloc(sizeof(double) * (size_t)D);
        double *g2 = malloc(sizeof(double) * (size_t)D);
        if (!s_buf || !g || !g2) {
#pragma omp atomic write
            failed = 1;
        }
        if (!failed) {
#pragma omp for schedule(dynamic, 4)
            for (int m = 0; m < L; m++) {
                if (!need[m])
                    continue;
                row_stats(qr, kr, v, dout, stride, D, scale, m, s_buf, &lse_all[m],
                          dout ? &delta_all[m] : NULL, NULL);
            }

            /* Query-row outputs: O_m, LSE_m, D_m, dq_m. */
#pragma omp for schedule(dynamic, 4)
            for (int i = 0; i < nq; i++) {
                int m = qrows[i];
                double lse_m = lse_all[m];
                if (lse)
                    lse[i] = lse_m;
                if (delta)
                    delta[i] = delta_all[m];
                if (o) {
                    double *om = o + (long long)i * D;
                    for (int d = 0; d < D; d++)
                        om[d] = 0.0;
                    for (int n = 0; n <= m; n++) {
                        double p = exp(scale * dot(qr + (long long)m * D, kr + (long long)n * D, D) - lse_m);
                        const double *vn = v + (long long)n * stride;
                        for (int d = 0; d < D; d++)
                            om[d] += p * vn[d];
                    }
                }
                if (dq) {
                    const double *dom = dout + (long long)m * stride;
                    for (int d = 0; d < D; d++)
                        g[d] = 0.0;
                    for (int n = 0; n <= m; n++) {
                        double p = exp(scale * dot(qr + (long long)m * D, kr + (long long)n * D, D) - lse_m);
                        double dp = dot(dom, v + (long long)n * stride, D);
                        double ds = p * (dp - delta_all[m]);
                        const double *kn = kr + (long long)n * D;
                        for (int d = 0; d < D; d++)
                            g[d] += ds * kn[d];
                    }
                    for (int d = 0; d < D; d++)
                        g[d] *= scale;
                    rope_vector_transpose(g, D, m, base, dq + (long long)i * D);
                }
            }

            /* Key-row outputs: dv_n, dk_n over all query rows m >= n. */
            if (dk || dv) {
#pragma omp for schedule(dynamic, 4)
                for (int i = 0; i < nk; i++) {
                    int n = krows[i];
                    for (int d = 0; d < D; d++) {
                        g[d] = 0.0;
                        g2[d] = 0.0;
                    }
                    const double *kn = kr + (long long)n * D;
                    const double *vn = v + (long long)n * stride;
                    for (int m = n; m < L; m++) {
                        const double *qm = qr + (long long)m * D;
                        const double *dom = dout + (long long)m * stride;
                        double p = exp(scale * dot(qm, kn, D) - lse_all[m]);
                        double dp = dot(dom, vn, D);
                        double ds = p * (dp - delta_all[m]);
                        for (int d = 0; d < D; d++) {
                            g[d] += ds * qm[d];   /* dk' before scale */
                            g2[d] += p * dom[d];  /* dv */
                        }
                    }
                    if (dv)
                        for (int d = 0; d < D; d++)
                            dv[(long long)i * D + d] = g2[d];
                    if (dk) {
                        for (int d = 0; d < D; d++)
                            g[d] *= scale;
                        rope_vector_transpose(g, D, n, base, dk + (long long)i * D);
                    }
                }
            }
        }
        free(s_buf);
        free(g);
        free(g2);
    }
    free(qr); free(kr); free(lse_all); free(delta_all); free(need);
    return failed ? -1 : 0;
}

/* Exported: the full probability matrix P[L][L] of one (sequence, head), for
 * the tests' row-sum and mask pins on tiny inputs. */
int ne_oracle_probs(const double *q, const double *k, long long stride, int L, int D,
                    double base, double scale, int mode, double *P)
{
    if (!q || !k || !P || L <= 0 || D <= 0 || (D % 2) != 0)
        return -1;
    double *qr = malloc(sizeof(double) * (size_t)L * D);
    double *kr = malloc(sizeof(double) * (size_t)L * D);
    double *s_buf = malloc(sizeof(double) * (size_t)L);
    if (!qr || !kr || !s_buf) {
        free(qr); free(kr); free(s_buf);
        return -1;
    }
    ne_oracle_rope(q, stride, L, D, base, mode, qr);
    ne_oracle_rope(k, stride, L, D, base, mode, kr);
    for (int m = 0; m < L; m++) {
        double lse;
        row_stats(qr, kr, NULL, NULL, stride, D, scale, m, s_buf, &lse, NULL, NULL);
        for (int n = 0; n < L; n++)
            P[(long long)m * L + n] = (n <= m) ? exp(s_buf[n] - lse) : 0.0;
    }
    free(qr); free(kr); free(s_buf);
    return 0;
}

/* Exported: number of OpenMP threads a parallel region here would use. */
int ne_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * ---- The projections around the attention (the step before and the step
 * after it in a transformer layer).  NanoEuler Show HN page, paragraph 2: the
 * CUDA engine has RMSNorm and RoPE kernels and computes the matrix products of
 * the layer; "Tiny Hackable CUDA", section 3: the projections are computed,
 * RoPE is applied to them to encode relative position, and the attention is
 * wrapped in a residual connection.  The pages print no equations; the
 * standard definitions are used (RMSNorm: Zhang and Sennrich 2019; linear
 * maps in the nn.Linear convention, weights [out, in], no bias):
 *
 *   RMSNorm:   xn[n][c] = x[n][c] / sqrt(mean_c' x[n][c']^2 + eps) * g[c]
 *   linear:    y[n][m]  = sum_k a[n][k] w[m][k]
 *   QKV:       [q | k | v] = linear(RMSNorm(x), w_qkv), w_qkv [3C, C];
 *              q', k' = R(t) q, R(t) k per head of D columns, at the token's
 *              position t within its sequence (rotate-half, as above)
 *   out proj:  y = r + linear(o, w_o), w_o [C, C]   (residual r)
 * Everything in double.
 */

/* Exported: RMSNorm of N rows of C.  Returns 0, or -1 on bad arguments. */
int ne_oracle_rmsnorm(const double *x, const double *g, int N, int C, double eps, double *out)
{
    if (!x || !g || !out || N < 0 || C <= 0 || !(eps >= 0.0))
        return -1;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const double *xr = x + (long long)n * C;
        double ss = 0.0;
        for (int c = 0; c < C; c++)
            ss += xr[c] * xr[c];
        double inv = 1.0 / sqrt(ss / C + eps);
        for (int c = 0; c < C; c++)
            out[(long long)n * C + c] = xr[c] * inv * g[c];
    }
    return 0;
}

/* Exported: y[N][M] = a[N][K] . w[M][K]^T.  Returns 0, or -1 on bad arguments. */
int ne_oracle_linear(const double *a, const double *w, int N, int K, int M, double *y)
{
    if (!a || !w || !y || N < 0 || K <= 0 || M <= 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++)
        for (int m = 0; m < M; m++)
            y[(long long)n * M + m] = dot(a + (long long)n * K, w + (long long)m * K, K);
    return 0;
}

/* Exported: the QKV projection with RoPE of a fixed-length batch of B
 * sequences of T tokens: x [B*T][C] (C = H*D), g [C], w [3C][C].  Writes
 * q', k', v [B*T][C] (head h in columns h*D .. h*D+D-1).  Returns 0, or -1. */
int ne_oracle_qkv_rope(const double *x, const double *g, const double *w, int B, int T, int H,
                       int D, double base, double eps, double *qr, double *kr, double *v)
{
    if (!x || !g || !w || !qr || !kr || !v || B <= 0 || T <= 0 || H <= 0 || D <= 0 || (D % 2))
        return -1;
    const int C = H * D;
    const long long N = (long long)B * T;
    double *xn = malloc(sizeof(double) * (size_t)N * C);
    double *y = malloc(sizeof(double) * (size_t)N * 3 * C);
    if (!xn || !y) {
        free(xn); free(y);
        return -1;
    }
    ne_oracle_rmsnorm(x, g, (int)N, C, eps, xn);
    ne_oracle_linear(xn, w, (int)N, C, 3 * C, y);
#pragma omp parallel for schedule(static)
    for (long long n = 0; n < N; n++) {
        const int t = (int)(n % T);
        const double *yr = y + n * 3 * C;
        for (int h = 0; h < H; h++) {
            rope_vector(yr + h * D, D, t, base, 0, qr + n * C + h * D);
            rope_vector(yr + C + h * D, D, t, base, 0, kr + n * C + h * D);
            for (int d = 0; d < D; d++)
                v[n * C + h * D + d] = yr[2 * C + h * D + d];
        }
    }
    free(xn);
    free(y);
    return 0;
}

/* Exported: y = r + o . w^T for N rows of C (w [C][C]).  Returns 0, or -1. */
int ne_oracle_out_proj_residual(const double *o, const double *w, const double *r, int N, int C,
                                double *y)
{
    if (!o || !w || !r || !y || N < 0 || C <= 0)
        return -1;
    if (ne_oracle_linear(o, w, N, C, C, y) != 0)
        return -1;
    for (long long i = 0; i < (long long)N * C; i++)
        y[i] += r[i];
    return 0;
}

/*
 * Multi-token prediction (MTP) head with its softmax cross-entropy loss and
 * analytic gradients (NanoEuler Show HN page, paragraph 2: the engine's
 * analytic gradients, "including the RoPE and MTP layers", are checked against
 * double-precision centred finite differences).  The page names the layers and
 * nothing more; the plainest reading is taken: K linear heads on the trunk's
 * hidden state h_t, head j (0-based) predicting the token j + 1 positions
 * ahead, each scored by softmax cross-entropy, the loss the mean over the
 * (t, j) with a target:
 *     logit_j(t)[v] = h_t . w_{jV+v}
 *     lse_j(t)      = log sum_v exp(logit_j(t)[v])
 *     loss          = (1/n) sum_{(t,j) with target} (lse_j(t) - logit_j(t)[y_tj])
 *     dlogit_j(t)   = (softmax(logit_j(t)) - onehot(y_tj)) / n
 *     dh_t          = sum_j sum_v dlogit_j(t)[v] w_{jV+v}
 *     dw_{jV+v}     = sum_t dlogit_j(t)[v] h_t
 * h [M][C], w [K*V][C], targets [M][K] (token id, or -1: no target there).
 * Writes loss (scalar; 0 when no (t, j) has a target), row_loss [M][K] (0
 * where there is no target), dh [M][C] and dw [K*V][C].  Returns 0, or -1.
 */
int ne_oracle_mtp_head(const double *h, const double *w, const int *targets, int M, int C, int K,
                       int V, double *loss, double *row_loss, double *dh, double *dw)
{
    if (!h || !w || !targets || !loss || !row_loss || !dh || !dw || M < 0 || C <= 0 || K <= 0 ||
        V <= 0)
        return -1;
    long long n = 0;
    for (long long i = 0; i < (long long)M * K; i++) {
        if (targets[i] >= V)
            return -1;
        if (targets[i] >= 0)
            n++;
    }
    for (long long i = 0; i < (long long)M * C; i++)
        dh[i] = 0.0;
    for (long long i = 0; i < (long long)K * V * C; i++)
        dw[i] = 0.0;
    double *logit = malloc(sizeof(double) * (size_t)V);
    if (!logit)
        return -1;
    double sum = 0.0;
    for (int t = 0; t < M; t++) {
        const double *ht = h + (long long)t * C;
        for (int j = 0; j < K; j++) {
            const int y = targets[(long long)t * K + j];
            row_loss[(long long)t * K + j] = 0.0;
            if (y < 0)
                continue;
            const double *wj = w + (long long)j * V * C;
            double mx = -INFINITY;
            for (int v = 0; v < V; v++) {
                logit[v] = dot(ht, wj + (long long)v * C, C);
                if (logit[v] > mx)
                    mx = logit[v];
            }
            double se = 0.0;
            for (int v = 0; v < V; v++)
                se += exp(logit[v] - mx);
            const double lse = mx + log(se);
            row_loss[(long long)t * K + j] = lse - logit[y];
            sum += lse - logit[y];
            for (int v = 0; v < V; v++) {
                const double g = (exp(logit[v] - lse) - (v == y ? 1.0 : 0.0)) / (double)n;
                const double *wv = wj + (long long)v * C;
                double *dwv = dw + ((long long)j * V + v) * C;
                for (int c = 0; c < C; c++) {
                    dh[(long long)t * C + c] += g * wv[c];
                    dwv[c] += g * ht[c];
                }
            }
        }
    }
    free(logit);
    *loss = n > 0 ? sum / (double)n : 0.0;
    return 0;
}

