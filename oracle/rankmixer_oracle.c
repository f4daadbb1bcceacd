/*
 * RankMixer CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct restatement of the RankMixer block forward
 * in double precision.  It exists to check the CUDA library; only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header or table with the CUDA path.
 *
 * Sources (the pages this restates):
 *   [RM]  "RankMixer: Scaling Up Ranking Models in Industrial Recommenders"
 *         (Zhu et al., ByteDance), section 3.1 Eq. 1, section 3.3.1 Eq. 3-5,
 *         section 3.3.2 Eq. 6-9, section 3.4 Eq. 10, section 3.5 Eq. 12.
 *   [TU]  "6.4 Rankmixer: 硬件效率优化", section 6.4.4 (DTSI-MoE routers).
 *   [UM]  "UniMixer: A Unified Architecture for Scaling Laws in
 *         Recommendation Systems", section 4.3 Eq. 11-15 (UniMixing and its
 *         constrained weights), Appendix A (the TokenMixer as a Kronecker
 *         product), Appendix B (the computation flow, Eq. 24-29).
 *   [WT]  "RankMixer 详解（1）：特征分组与完整计算流程", section 3.1 (the
 *         element map of TokenMixing), section 3.3 (LayerNorm definition),
 *         section 4.1 (GELU = u*Phi(u), row-vector FFN), section 5.1 (mean
 *         pooling).
 *
 * Conventions (all arrays row-major, double):
 *   X      [B][T][D]        token matrix per sample
 *   W1     [T][D][F]        per-token first layer, u = s W1 + b1   (F = kD)
 *   b1     [T][F]
 *   W2     [T][F][D]        per-token second layer, v = a W2 + b2
 *   b2     [T][D]
 *   g1,be1,g2,be2 [D]       LayerNorm affine, one pair per LN, shared by tokens
 *
 * Every function is a direct loop nest over the definition.  The only
 * concession to speed is an OpenMP loop over independent samples.
 */
#include <math.h>
#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#if defined(_OPENMP)
#include <omp.h>
#endif

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------ */
/* TokenMixing, [RM] Eq. 3-4 and [WT] section 3.1:                     */
/*   SplitHead cuts each token x_t into H contiguous blocks of q = D/H; */
/*   mixed row h is Concat(x_1^h, ..., x_T^h), so                       */
/*   M[h][t*q + r] = X[t][h*q + r]   (0-based t, h, r).                 */
/* Output is [H][T*q]; with H = T it has the input's shape [T][D].      */
/* ------------------------------------------------------------------ */
static void mix_sample(const double *X, double *M, int T, int D, int H)
{
    const int q = D / H;
    for (int h = 0; h < H; ++h)
        for (int t = 0; t < T; ++t)
            for (int r = 0; r < q; ++r)
                M[(size_t)h * T * q + (size_t)t * q + r] = X[(size_t)t * D + (size_t)h * q + r];
}

ORACLE_API void oracle_token_mix(const double *X, double *M, int B, int T, int D, int H)
{
    const size_t per = (size_t)T * D;
    for (int b = 0; b < B; ++b)
        mix_sample(X + b * per, M + b * per, T, D, H);
}

/* ------------------------------------------------------------------ */
/* LayerNorm over one row of length D, [WT] section 3.3:               */
/*   mu = (1/D) sum r_j,  var = (1/D) sum (r_j - mu)^2  (biased),       */
/*   out_j = gamma_j (r_j - mu) / sqrt(var + eps) + beta_j.             */
/* ------------------------------------------------------------------ */
static void layernorm_row(const double *r, const double *gamma, const double *beta,
                          double eps, double *out, int D)
{
    double mu = 0.0;
    for (int j = 0; j < D; ++j) mu += r[j];
    mu /= (double)D;
    double var = 0.0;
    for (int j = 0; j < D; ++j) var += (r[j] - mu) * (r[j] - mu);
    var /= (double)D;
    const double inv = 1.0 / sqrt(var + eps);
    for (int j = 0; j < D; ++j) out[j] = gamma[j] * (r[j] - mu) * inv + beta[j];
}

ORACLE_API void oracle_layernorm(const double *R, const double *gamma, const double *beta,
                                 double eps, double *out, int rows, int D)
{
    for (int i = 0; i < rows; ++i)
        layernorm_row(R + (size_t)i * D, gamma, beta, eps, out + (size_t)i * D, D);
}

/* GELU, [WT] section 4.1: Gelu(u) = u * Phi(u), Phi the standard normal CDF,
 * Phi(u) = (1 + erf(u / sqrt 2)) / 2. */
static double gelu(double u)
{
    return u * 0.5 * (1.0 + erf(u / sqrt(2.0)));
}

ORACLE_API void oracle_gelu(const double *u, double *out, size_t n)
{
    for (size_t i = 0; i < n; ++i) out[i] = gelu(u[i]);
}

/* One two-layer FFN on a row vector, [RM] Eq. 6-7:
 *   u = s W1 + b1 (length F), a = Gelu(u), v = a W2 + b2 (length D).
 * Each output starts from its bias and adds the products in ascending input
 * index; the loops run over W's rows so the matrices are read in order. */
static void ffn_row(const double *s, const double *W1, const double *b1,
                    const double *W2, const double *b2, double *v, double *a_scratch,
                    int D, int F)
{
    for (int j = 0; j < F; ++j) a_scratch[j] = b1[j];
    for (int i = 0; i < D; ++i) {
        const double si = s[i];
        const double *w = W1 + (size_t)i * F;
        for (int j = 0; j < F; ++j) a_scratch[j] += si * w[j];
    }
    for (int j = 0; j < F; ++j) a_scratch[j] = gelu(a_scratch[j]);
    for (int j = 0; j < D; ++j) v[j] = b2[j];
    for (int i = 0; i < F; ++i) {
        const double ai = a_scratch[i];
        const double *w = W2 + (size_t)i * D;
        for (int j = 0; j < D; ++j) v[j] += ai * w[j];
    }
}

/* Per-token FFN on one sample, [RM] Eq. 8-9: token t uses its own weights. */
ORACLE_API void oracle_pffn(const double *S, const double *W1, const double *b1,
                            const double *W2, const double *b2, double *V,
                            int B, int T, int D, int F)
{
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * (size_t)F);
#pragma omp for schedule(static)
        for (int b = 0; b < B; ++b)
            for (int t = 0; t < T; ++t) {
                const size_t row = ((size_t)b * T + t) * D;
                ffn_row(S + row, W1 + (size_t)t * D * F, b1 + (size_t)t * F,
                        W2 + (size_t)t * F * D, b2 + (size_t)t * D, V + row, a, D, F);
            }
        free(a);
    }
}

/* ------------------------------------------------------------------ */
/* UniMixing, [UM] section 4.3.                                        */
/*                                                                    */
/* Constrained weights, Eq. 15: each n x n matrix W is symmetrised,     */
/* W~ = (W + W^T) / 2, and handed to Sinkhorn-Knopp at temperature tau: */
/* every element becomes exp(W~ / tau) (positive), then `iters` rounds  */
/* each divide every row by its sum and then every column by its sum.   */
/* The pages fix neither the round count nor which axis goes first;     */
/* here a round is rows, then columns.                                  */
/* ------------------------------------------------------------------ */
ORACLE_API void oracle_sinkhorn(const double *W, double *out, int count, int n, double tau, int iters)
{
    const size_t nn = (size_t)n * n;
    for (int c = 0; c < count; ++c) {
        const double *w = W + (size_t)c * nn;
        double *o = out + (size_t)c * nn;
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j)
                o[(size_t)i * n + j] = exp(0.5 * (w[(size_t)i * n + j] + w[(size_t)j * n + i]) / tau);
        for (int it = 0; it < iters; ++it) {
            for (int i = 0; i < n; ++i) {
                double sum = 0.0;
                for (int j = 0; j < n; ++j) sum += o[(size_t)i * n + j];
                for (int j = 0; j < n; ++j) o[(size_t)i * n + j] /= sum;
            }
            for (int j = 0; j < n; ++j) {
                double sum = 0.0;
                for (int i = 0; i < n; ++i) sum += o[(size_t)i * n + j];
                for (int i = 0; i < n; ++i) o[(size_t)i * n + j] /= sum;
            }
        }
    }
}

/* UniMixing of one flattened sample, [UM] Eq. 12-14 (the optimised flow,  */
/* Appendix B Eq. 29): flatten(X) (length L) is cut into nb = L / bs row   */
/* vectors x_j; the local step is h_j = x_j WB_j (bs x bs, one per block); */
/* the global step is out_i = sum_j WG[i][j] h_j; the output is            */
/* out_0 | out_1 | ... | out_{nb-1}, reshaped back to X's shape.           */
/* WG [nb][nb], WB [nb][bs][bs] (row s, column r), h: nb * bs scratch.     */
static void unimix_sample(const double *x, double *y, const double *WG, const double *WB, int L, int bs,
                          double *h)
{
    const int nb = L / bs;
    for (int j = 0; j < nb; ++j)
        for (int r = 0; r < bs; ++r) {
            double acc = 0.0;
            for (int s = 0; s < bs; ++s)
                acc += x[(size_t)j * bs + s] * WB[((size_t)j * bs + s) * bs + r];
            h[(size_t)j * bs + r] = acc;
        }
    for (int i = 0; i < nb; ++i)
        for (int r = 0; r < bs; ++r) {
            double acc = 0.0;
            for (int j = 0; j < nb; ++j) acc += WG[(size_t)i * nb + j] * h[(size_t)j * bs + r];
            y[(size_t)i * bs + r] = acc;
        }
}

/* Y[b] = UniMixing(X[b]) for B samples of length L (block size bs). */
ORACLE_API void oracle_unimixing(const double *X, double *Y, const double *WG, const double *WB, int B, int L,
                                 int bs)
{
#pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)L);
#pragma omp for schedule(static)
        for (int b = 0; b < B; ++b)
            unimix_sample(X + (size_t)b * L, Y + (size_t)b * L, WG, WB, L, bs, h);
        free(h);
    }
}

/* ------------------------------------------------------------------ */
/* One RankMixer block on one sample, [RM] Eq. 1:                       */
/*   S  = LN1(TokenMixing(X) + X)                                       */
/*   X' = LN2(PFFN(S) + S)                                              */
/* S_out may be NULL.  Requires H = T (the residual needs equal shape). */
/* With WG non-NULL the mixing is UniMixing with constrained weights    */
/* WG, WB and block size bs ([UM] Eq. 14) in place of TokenMixing; the  */
/* rest of the block is unchanged.                                      */
/* ------------------------------------------------------------------ */
static void block_sample(const double *X, double *Xout, double *S_keep,
                         const double *W1, const double *b1, const double *W2, const double *b2,
                         const double *g1, const double *be1, const double *g2, const double *be2,
                         const double *WG, const double *WB, int bs,
                         double eps, int T, int D, int F, double *work)
{
    const size_t TD = (size_t)T * D;
    double *M = work;            /* [T][D] mixed   */
    double *S = M + TD;          /* [T][D] LN1 out */
    double *Y = S + TD;          /* [T][D] residual sums */
    double *hb = Y + TD;         /* [T*D] UniMixing local outputs */
    double *a = hb + TD;         /* [F]   hidden   */
    double *v = a + F;           /* [D]   FFN out  */

    if (WG)
        unimix_sample(X, M, WG, WB, (int)TD, bs, hb);
    else
        mix_sample(X, M, T, D, T);
    for (size_t i = 0; i < TD; ++i) Y[i] = M[i] + X[i];
    for (int t = 0; t < T; ++t) layernorm_row(Y + (size_t)t * D, g1, be1, eps, S + (size_t)t * D, D);

    for (int t = 0; t < T; ++t) {
        ffn_row(S + (size_t)t * D, W1 + (size_t)t * D * F, b1 + (size_t)t * F,
                W2 + (size_t)t * F * D, b2 + (size_t)t * D, v, a, D, F);
        for (int j = 0; j < D; ++j) Y[(size_t)t * D + j] = v[j] + S[(size_t)t * D + j];
        layernorm_row(Y + (size_t)t * D, g2, be2, eps, Xout + (size_t)t * D, D);
    }
    if (S_keep) memcpy(S_keep, S, sizeof(double) * TD);
}

ORACLE_API void oracle_block_forward(const double *X, double *Xout, double *S_out,
                                     const double *W1, const double *b1,
                                     const double *W2, const double *b2,
                                     const double *g1, const double *be1,
                                     const double *g2, const double *be2,
                                     double eps, int B, int T, int D, int F)
{
    const size_t TD = (size_t)T * D;
#pragma omp parallel
    {
        double *work = (double *)malloc(sizeof(double) * (4 * TD + (size_t)F + (size_t)D));
#pragma omp for schedule(static)
        for (int b = 0; b < B; ++b)
            block_sample(X + b * TD, Xout + b * TD, S_out ? S_out + b * TD : NULL,
                         W1, b1, W2, b2, g1, be1, g2, be2, NULL, NULL, 0, eps, T, D, F, work);
        free(work);
    }
}

/* Mean pooling, [RM] section 3.1 / [WT] section 5.1: o = (1/T) sum_t X_L[t,:]. */
ORACLE_API void oracle_mean_pool(const double *X, double *o, int B, int T, int D)
{
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < D; ++j) {
            double acc = 0.0;
            for (int t = 0; t < T; ++t) acc += X[((size_t)b * T + t) * D + j];
            o[(size_t)b * D + j] = acc / (double)T;
        }
}

/* ------------------------------------------------------------------ */
/* L stacked blocks with independent per-layer weights ([RM] Eq. 1 and  */
/* the factor L in Eq. 12), then mean pooling.  Per-layer parameter     */
/* arrays are concatenated along a leading layer axis.  XL may be NULL. */
/* ------------------------------------------------------------------ */
static void stack_forward(const double *X0, double *pooled, double *XL,
                          const double *W1, const double *b1,
                          const double *W2, const double *b2,
                          const double *g1, const double *be1,
                          const double *g2, const double *be2,
                          const double *WG, const double *WB, int bs,
                          double eps, int B, int T, int D, int F, int L)
{
    const size_t TD = (size_t)T * D;
#pragma omp parallel
    {
        double *work = (double *)malloc(sizeof(double) * (4 * TD + (size_t)F + (size_t)D));
        double *cur = (double *)malloc(sizeof(double) * TD);
        double *nxt = (double *)malloc(sizeof(double) * TD);
#pragma omp for schedule(static)
        for (int b = 0; b < B; ++b) {
            memcpy(cur, X0 + b * TD, sizeof(double) * TD);
            for (int n = 0; n < L; ++n) {
                block_sample(cur, nxt, NULL,
                             W1 + (size_t)n * T * D * F, b1 + (size_t)n * T * F,
                             W2 + (size_t)n * T * F * D, b2 + (size_t)n * T * D,
                             g1 + (size_t)n * D, be1 + (size_t)n * D,
                             g2 + (size_t)n * D, be2 + (size_t)n * D,
                             WG ? WG + (size_t)n * (T * D / bs) * (T * D / bs) : NULL,
                             WB ? WB + (size_t)n * T * D * bs : NULL, bs, eps, T, D, F, work);
                double *tmp = cur; cur = nxt; nxt = tmp;
            }
            for (int j = 0; j < D; ++j) {
                double acc = 0.0;
                for (int t = 0; t < T; ++t) acc += cur[(size_t)t * D + j];
                pooled[(size_t)b * D + j] = acc / (double)T;
            }
            if (XL) memcpy(XL + b * TD, cur, sizeof(double) * TD);
        }
        free(work); free(cur); free(nxt);
    }
}

ORACLE_API void oracle_stack_forward(const double *X0, double *pooled, double *XL,
                                     const double *W1, const double *b1,
                                     const double *W2, const double *b2,
                                     const double *g1, const double *be1,
                                     const double *g2, const double *be2,
                                     double eps, int B, int T, int D, int F, int L)
{
    stack_forward(X0, pooled, XL, W1, b1, W2, b2, g1, be1, g2, be2, NULL, NULL, 0, eps, B, T, D, F, L);
}

/* The stack with UniMixing in every layer ([UM] Eq. 14 in place of [RM]   */
/* Eq. 3-4): WG [L][nb][nb] and WB [L][nb][bs][bs] are the constrained      */
/* weights (see oracle_sinkhorn), nb = T * D / bs.                          */
ORACLE_API void oracle_stack_forward_unimix(const double *X0, double *pooled, double *XL,
                                            const double *W1, const double *b1,
                                            const double *W2, const double *b2,
                                            const double *g1, const double *be1,
                                            const double *g2, const double *be2,
                                            const double *WG, const double *WB, int bs,
                                            double eps, int B, int T, int D, int F, int L)
{
    stack_forward(X0, pooled, XL, W1, b1, W2, b2, g1, be1, g2, be2, WG, WB, bs, eps, B, T, D, F, L);
}

/* ------------------------------------------------------------------ */
/* Sparse-MoE PFFN with ReLU routing, [RM] section 3.4 Eq. 10:          */
/*   G[t][e] = ReLU(h_t(s_t))  with the inference router h_t linear:   */
/*             h_t(s) = s Wg_t + bg_t,  Wg_t [D][E], bg_t [E];          */
/*   v_t = sum_e G[t][e] * FFN_{t,e}(s_t), every expert a two-layer     */
/*   GELU FFN D -> Fe -> D owned by token t alone.                      */
/* All experts are evaluated densely; a zero gate contributes exactly 0.*/
/*   S [B][T][D], Wg [T][D][E], bg [T][E], eW1 [T][E][D][Fe],           */
/*   eb1 [T][E][Fe], eW2 [T][E][Fe][D], eb2 [T][E][D];                  */
/*   V [B][T][D], G [B][T][E] (G may be NULL).                          */
/* ------------------------------------------------------------------ */
ORACLE_API void oracle_moe_pffn(const double *S, const double *Wg, const double *bg,
                                const double *eW1, const double *eb1,
                                const double *eW2, const double *eb2,
                                double *V, double *G, int B, int T, int D, int E, int Fe)
{
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * (size_t)Fe);
        double *v = (double *)malloc(sizeof(double) * (size_t)D);
        double *g = (double *)malloc(sizeof(double) * (size_t)E);
#pragma omp for schedule(static)
        for (int b = 0; b < B; ++b)
            for (int t = 0; t < T; ++t) {
                const double *s = S + ((size_t)b * T + t) * D;
                double *out = V + ((size_t)b * T + t) * D;
                for (int e = 0; e < E; ++e) {
                    double h = bg[(size_t)t * E + e];
                    for (int i = 0; i < D; ++i) h += s[i] * Wg[((size_t)t * D + i) * E + e];
                    g[e] = h > 0.0 ? h : 0.0;
                    if (G) G[((size_t)b * T + t) * E + e] = g[e];
                }
                for (int j = 0; j < D; ++j) out[j] = 0.0;
                for (int e = 0; e < E; ++e) {
                    const size_t te = (size_t)t * E + e;
                    ffn_row(s, eW1 + te * D * Fe, eb1 + te * Fe, eW2 + te * Fe * D, eb2 + te * D,
                            v, a, D, Fe);
                    for (int j = 0; j < D; ++j) out[j] += g[e] * v[j];
                }
            }
        free(a); free(v); free(g);
    }
}

/* ================================================================== */
/* Backward pass of one block, "RankMixer 详解（1）" section 5.2.        */
/* ================================================================== */

/* Gelu'(u) = Phi(u) + u phi(u), phi the standard normal density        */
/* ([WT] section 5.2, derivative of the exact GELU).                   */
static double gelu_grad(double u)
{
    const double Phi = 0.5 * (1.0 + erf(u / sqrt(2.0)));
    const double phi = exp(-0.5 * u * u) / sqrt(2.0 * M_PI);
    return Phi + u * phi;
}

ORACLE_API void oracle_gelu_grad(const double *u, double *out, size_t n)
{
    for (size_t i = 0; i < n; ++i) out[i] = gelu_grad(u[i]);
}

/* LayerNorm backward on one row ([WT] section 5.2).  r is the LN input, */
/* g the gradient arriving at the LN output:                          */
/*   rhat_j = (r_j - mu) / sqrt(var + eps),  q_j = g_j gamma_j,         */
/*   dr_j = (q_j - mean(q) - rhat_j mean(q rhat)) / sqrt(var + eps),    */
/* and the affine parameters receive g_j rhat_j (gamma) and g_j (beta), */
/* added into dgamma / dbeta when those are not NULL.                  */
static void layernorm_row_backward(const double *r, const double *gamma, const double *g, double eps,
                                   double *dr, double *dgamma, double *dbeta, int D)
{
    double mu = 0.0;
    for (int j = 0; j < D; ++j) mu += r[j];
    mu /= (double)D;
    double var = 0.0;
    for (int j = 0; j < D; ++j) var += (r[j] - mu) * (r[j] - mu);
    var /= (double)D;
    const double inv = 1.0 / sqrt(var + eps);
    double mq = 0.0, mqr = 0.0;
    for (int j = 0; j < D; ++j) {
        const double rh = (r[j] - mu) * inv;
        const double qj = g[j] * gamma[j];
        mq += qj;
        mqr += qj * rh;
    }
    mq /= (double)D;
    mqr /= (double)D;
    for (int j = 0; j < D; ++j) {
        const double rh = (r[j] - mu) * inv;
        dr[j] = (g[j] * gamma[j] - mq - rh * mqr) * inv;
        if (dgamma) dgamma[j] += g[j] * rh;
        if (dbeta) dbeta[j] += g[j];
    }
}

ORACLE_API void oracle_layernorm_backward(const double *R, const double *gamma, const double *Gout, double eps,
                                          double *dR, double *dgamma, double *dbeta, int rows, int D)
{
    for (int j = 0; j < D; ++j) dgamma[j] = dbeta[j] = 0.0;
    for (int i = 0; i < rows; ++i)
        layernorm_row_backward(R + (size_t)i * D, gamma, Gout + (size_t)i * D, eps, dR + (size_t)i * D,
                               dgamma, dbeta, D);
}

/* ------------------------------------------------------------------ */
/* Block backward.  Given the block input X and G = dl/dX' at its output */
/* (X' = LN2(PFFN(S) + S), S = LN1(Mix(X) + X), [RM] Eq. 1), returns     */
/* dX = dl/dX and the parameter gradients summed over the batch.        */
/* For row (b, t), with u = s W1 + b1, a = Gelu(u), z = a W2 + b2 + s:  */
/*   dz  = LN2 backward of G[b,t]          (also the residual's share)  */
/*   dW2 += a^T dz,  db2 += dz,  da = dz W2^T                          */
/*   du  = da * Gelu'(u)                                                */
/*   dW1 += s^T du,  db1 += du,  ds = du W1^T + dz                      */
/*   dy  = LN1 backward of ds              (y = Mix(X)[t] + X[t])       */
/* and finally dX = P^T dY + dY with P the mixing permutation           */
/* ([WT] section 5.2: the transpose routes each coordinate back).       */
/* Rows of one token only touch that token's weights, so the loop runs  */
/* tokens in parallel and samples in order: the sums over b do not      */
/* depend on the thread count.  Requires H = T.                         */
/* ------------------------------------------------------------------ */
ORACLE_API void oracle_block_backward(const double *X, const double *G, double *dX,
                                      const double *W1, const double *b1, const double *W2, const double *b2,
                                      const double *g1, const double *be1, const double *g2, const double *be2,
                                      double eps,
                                      double *dW1, double *db1, double *dW2, double *db2,
                                      double *dg1, double *dbe1, double *dg2, double *dbe2,
                                      int B, int T, int D, int F)
{
    const int q = D / T;
    const size_t TD = (size_t)T * D;
    double *dY = (double *)malloc(sizeof(double) * (size_t)B * TD);
    /* per-token partial sums of the LayerNorm affine gradients */
    double *pg1 = (double *)calloc(TD, sizeof(double));
    double *pbe1 = (double *)calloc(TD, sizeof(double));
    double *pg2 = (double *)calloc(TD, sizeof(double));
    double *pbe2 = (double *)calloc(TD, sizeof(double));
    memset(dW1, 0, sizeof(double) * TD * F);
    memset(db1, 0, sizeof(double) * (size_t)T * F);
    memset(dW2, 0, sizeof(double) * TD * F);
    memset(db2, 0, sizeof(double) * TD);

#pragma omp parallel
    {
        double *y = (double *)malloc(sizeof(double) * (size_t)(6 * D + 4 * F));
        double *s = y + D, *z = s + D, *dz = z + D, *ds = dz + D, *dy = ds + D;
        double *u = dy + D, *a = u + F, *da = a + F, *du = da + F;
#pragma omp for schedule(dynamic, 1)
        for (int t = 0; t < T; ++t) {
            const double *W1t = W1 + (size_t)t * D * F, *b1t = b1 + (size_t)t * F;
            const double *W2t = W2 + (size_t)t * F * D, *b2t = b2 + (size_t)t * D;
            double *dW1t = dW1 + (size_t)t * D * F, *db1t = db1 + (size_t)t * F;
            double *dW2t = dW2 + (size_t)t * F * D, *db2t = db2 + (size_t)t * D;
            for (int b = 0; b < B; ++b) {
                const double *x = X + (size_t)b * TD;
                /* forward of row (b, t): Mix(X)[t][c q + r] = X[c][t q + r] */
                for (int c = 0; c < T; ++c)
                    for (int r = 0; r < q; ++r)
                        y[c * q + r] = x[(size_t)c * D + (size_t)t * q + r] + x[(size_t)t * D + (size_t)c * q + r];
                layernorm_row(y, g1, be1, eps, s, D);
                for (int j = 0; j < F; ++j) u[j] = b1t[j];
                for (int i = 0; i < D; ++i)
                    for (int j = 0; j < F; ++j) u[j] += s[i] * W1t[(size_t)i * F + j];
                for (int j = 0; j < F; ++j) a[j] = gelu(u[j]);
                for (int j = 0; j < D; ++j) z[j] = b2t[j] + s[j];
                for (int i = 0; i < F; ++i)
                    for (int j = 0; j < D; ++j) z[j] += a[i] * W2t[(size_t)i * D + j];
                /* backward */
                layernorm_row_backward(z, g2, G + (size_t)b * TD + (size_t)t * D, eps, dz,
                                       pg2 + (size_t)t * D, pbe2 + (size_t)t * D, D);
                for (int i = 0; i < F; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < D; ++j) {
                        dW2t[(size_t)i * D + j] += a[i] * dz[j];
                        acc += dz[j] * W2t[(size_t)i * D + j];
                    }
                    da[i] = acc;
                }
                for (int j = 0; j < D; ++j) db2t[j] += dz[j];
                for (int j = 0; j < F; ++j) {
                    du[j] = da[j] * gelu_grad(u[j]);
                    db1t[j] += du[j];
                }
                for (int i = 0; i < D; ++i) {
                    double acc = dz[i];
                    for (int j = 0; j < F; ++j) {
                        dW1t[(size_t)i * F + j] += s[i] * du[j];
                        acc += du[j] * W1t[(size_t)i * F + j];
                    }
                    ds[i] = acc;
                }
                layernorm_row_backward(y, g1, ds, eps, dy, pg1 + (size_t)t * D, pbe1 + (size_t)t * D, D);
                memcpy(dY + (size_t)b * TD + (size_t)t * D, dy, sizeof(double) * D);
            }
        }
        free(y);
    }
    /* dX = dY + P^T dY:  dX[t][c q + r] = dY[t][c q + r] + dY[c][t q + r] */
    for (int b = 0; b < B; ++b) {
        const double *g = dY + (size_t)b * TD;
        double *o = dX + (size_t)b * TD;
        for (int t = 0; t < T; ++t)
            for (int c = 0; c < T; ++c)
                for (int r = 0; r < q; ++r)
                    o[(size_t)t * D + c * q + r] = g[(size_t)t * D + c * q + r] + g[(size_t)c * D + (size_t)t * q + r];
    }
    for (int j = 0; j < D; ++j) {
        double s1 = 0.0, s2 = 0.0, s3 = 0.0, s4 = 0.0;
        for (int t = 0; t < T; ++t) {
            s1 += pg1[(size_t)t * D + j];
            s2 += pbe1[(size_t)t * D + j];
            s3 += pg2[(size_t)t * D + j];
            s4 += pbe2[(size_t)t * D + j];
        }
        dg1[j] = s1; dbe1[j] = s2; dg2[j] = s3; dbe2[j] = s4;
    }
    free(dY); free(pg1); free(pbe1); free(pg2); free(pbe2);
}

/* ------------------------------------------------------------------ */
/* Backward of L stacked blocks and the mean pool.  The pool hands each */
/* token row the same share, dl/dX_L[t] = g_o / T ([WT] section 5.2);   */
/* the blocks then run in reverse order, each fed its saved input.      */
/* Gradient arrays are concatenated along a leading layer axis.         */
/* ------------------------------------------------------------------ */
ORACLE_API void oracle_stack_backward(const double *X0, const double *dpooled, double *dX0,
                                      const double *W1, const double *b1, const double *W2, const double *b2,
                                      const double *g1, const double *be1, const double *g2, const double *be2,
                                      double eps,
                                      double *dW1, double *db1, double *dW2, double *db2,
                                      double *dg1, double *dbe1, double *dg2, double *dbe2,
                                      int B, int T, int D, int F, int L)
{
    const size_t TD = (size_t)T * D, BTD = (size_t)B * TD;
    double *Xs = (double *)malloc(sizeof(double) * BTD * (size_t)L);   /* input of each layer */
    double *Gc = (double *)malloc(sizeof(double) * BTD);
    double *Gn = (double *)malloc(sizeof(double) * BTD);
    memcpy(Xs, X0, sizeof(double) * BTD);
    for (int n = 0; n + 1 < L; ++n)
        oracle_block_forward(Xs + (size_t)n * BTD, Xs + (size_t)(n + 1) * BTD, NULL,
                             W1 + (size_t)n * TD * F, b1 + (size_t)n * T * F,
                             W2 + (size_t)n * TD * F, b2 + (size_t)n * TD,
                             g1 + (size_t)n * D, be1 + (size_t)n * D, g2 + (size_t)n * D, be2 + (size_t)n * D,
                             eps, B, T, D, F);
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < D; ++j) Gc[(size_t)b * TD + (size_t)t * D + j] = dpooled[(size_t)b * D + j] / (double)T;
    for (int n = L - 1; n >= 0; --n) {
        oracle_block_backward(Xs + (size_t)n * BTD, Gc, n == 0 ? dX0 : Gn,
                              W1 + (size_t)n * TD * F, b1 + (size_t)n * T * F,
                              W2 + (size_t)n * TD * F, b2 + (size_t)n * TD,
                              g1 + (size_t)n * D, be1 + (size_t)n * D, g2 + (size_t)n * D, be2 + (size_t)n * D, eps,
                              dW1 + (size_t)n * TD * F, db1 + (size_t)n * T * F,
                              dW2 + (size_t)n * TD * F, db2 + (size_t)n * TD,
                              dg1 + (size_t)n * D, dbe1 + (size_t)n * D, dg2 + (size_t)n * D, dbe2 + (size_t)n * D,
                              B, T, D, F);
        double *tmp = Gc; Gc = Gn; Gn = tmp;
    }
    free(Xs); free(Gc); free(Gn);
}

/* ------------------------------------------------------------------ */
/* Prediction head on the pooled output, [WT] sections 5.1-5.2:         */
/*   z = o w + b,  p = sigmoid(z) = 1 / (1 + e^-z),                     */
/*   l = -y log p - (1 - y) log(1 - p),  dl/dz = p - y,                 */
/*   dl/do = (p - y) w.                                                 */
/* log p = -softplus(-z) and log(1 - p) = -softplus(z) with             */
/* softplus(x) = log(1 + e^x), written so neither overflows.            */
/* y, loss, dz and dO may be NULL (no label: z and p only).             */
/* ------------------------------------------------------------------ */
static double softplus(double x)
{
    return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

ORACLE_API void oracle_head(const double *O, const double *w, double b, const double *y,
                            double *z, double *p, double *loss, double *dz, double *dO, int B, int D)
{
    for (int i = 0; i < B; ++i) {
        double zi = b;
        for (int j = 0; j < D; ++j) zi += O[(size_t)i * D + j] * w[j];
        const double pi = 1.0 / (1.0 + exp(-zi));
        if (z) z[i] = zi;
        if (p) p[i] = pi;
        if (!y) continue;
        if (loss) loss[i] = y[i] * softplus(-zi) + (1.0 - y[i]) * softplus(zi);
        if (dz) dz[i] = pi - y[i];
        if (dO)
            for (int j = 0; j < D; ++j) dO[(size_t)i * D + j] = (pi - y[i]) * w[j];
    }
}

/* ------------------------------------------------------------------ */
/* Feature tokenization, [RM] Eq. 2 / [WT] section 2.4: token i is the  */
/* i-th slice of d coordinates of the concatenated embedding, projected */
/* to D by its own linear layer,                                        */
/*   x_i = e[d (i-1) : d i] W_i + b_i,  W_i [d][D], b_i [D]             */
/* (0-based here: slice t is e[t d : (t + 1) d]).  E [B][T d] -> X0     */
/* [B][T][D].  Backward: dW_i = sum_b e_slice^T dX0[b][i],              */
/* db_i = sum_b dX0[b][i], dE slice = dX0[b][i] W_i^T.                  */
/* ------------------------------------------------------------------ */
ORACLE_API void oracle_tokenize(const double *E, const double *W, const double *bias, double *X0,
                                int B, int T, int d, int D)
{
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            const double *e = E + (size_t)b * T * d + (size_t)t * d;
            double *x = X0 + ((size_t)b * T + t) * D;
            for (int j = 0; j < D; ++j) x[j] = bias[(size_t)t * D + j];
            for (int i = 0; i < d; ++i)
                for (int j = 0; j < D; ++j) x[j] += e[i] * W[((size_t)t * d + i) * D + j];
        }
}

ORACLE_API void oracle_tokenize_backward(const double *E, const double *W, const double *dX0, double *dE,
                                         double *dW, double *db, int B, int T, int d, int D)
{
    memset(dW, 0, sizeof(double) * (size_t)T * d * D);
    memset(db, 0, sizeof(double) * (size_t)T * D);
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            const double *e = E + (size_t)b * T * d + (size_t)t * d;
            const double *g = dX0 + ((size_t)b * T + t) * D;
            double *de = dE + (size_t)b * T * d + (size_t)t * d;
            for (int j = 0; j < D; ++j) db[(size_t)t * D + j] += g[j];
            for (int i = 0; i < d; ++i) {
                double acc = 0.0;
                for (int j = 0; j < D; ++j) {
                    dW[((size_t)t * d + i) * D + j] += e[i] * g[j];
                    acc += g[j] * W[((size_t)t * d + i) * D + j];
                }
                de[i] = acc;
            }
        }
}

/* ------------------------------------------------------------------ */
/* Training forward of the Sparse-MoE PFFN, dense-training / sparse-    */
/* inference ([RM] section 3.4 Eq. 10-11; [TU] section 6.4.4 Eq. 6.4.7):*/
/* two linear routers per token, h_train and h_infer; the forward uses  */
/*   G_train = ReLU(s Wt_t + bt_t),  v = sum_e G_train[e] FFN_{t,e}(s), */
/* and alongside it G_infer = ReLU(s Wi_t + bi_t), whose sum is the     */
/* sparsity regulariser: L_reg[b] = sum_{t,e} G_infer[b,t,e] per sample */
/* (Eq. 11 sums over tokens i and experts j) and the per-expert         */
/* activation A[e] = sum_{b,t} G_infer[b,t,e] over the batch.           */
/* G_train, G_infer [B][T][E]; lreg [B]; A [E].                         */
/* ------------------------------------------------------------------ */
ORACLE_API void oracle_moe_pffn_train(const double *S, const double *Wt, const double *bt,
                                      const double *Wi, const double *bi,
                                      const double *eW1, const double *eb1, const double *eW2, const double *eb2,
                                      double *V, double *Gtrain, double *Ginfer, double *lreg, double *A,
                                      int B, int T, int D, int E, int Fe)
{
    oracle_moe_pffn(S, Wt, bt, eW1, eb1, eW2, eb2, V, Gtrain, B, T, D, E, Fe);
    for (int e = 0; e < E; ++e) A[e] = 0.0;
    for (int b = 0; b < B; ++b) {
        double l = 0.0;
        for (int t = 0; t < T; ++t) {
            const double *s = S + ((size_t)b * T + t) * D;
            for (int e = 0; e < E; ++e) {
                double h = bi[(size_t)t * E + e];
                for (int i = 0; i < D; ++i) h += s[i] * Wi[((size_t)t * D + i) * E + e];
                const double g = h > 0.0 ? h : 0.0;
                Ginfer[((size_t)b * T + t) * E + e] = g;
                l += g;
                A[e] += g;
            }
        }
        lreg[b] = l;
    }
}

ORACLE_API int oracle_num_threads(void)
{
#if defined(_OPENMP)
    return omp_get_max_threads();
#else
    return 1;
#endif
}

ORACLE_API void oracle_set_num_threads(int n)
{
#if defined(_OPENMP)
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
