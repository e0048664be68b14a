/*
 * moe_oracle.c -- plain CPU oracle of the group-limited MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline / reference legs of bench.py may load or call this code.  The
 * CUDA library never links it and shares no code, header, table or helper
 * with it.  It is deliberately slow: plain loops, double accumulation, and a
 * single rounding to fp32 wherever the method fixes fp32.
 *
 * What it follows.  "The routing page" is the article
 *   "InternLumina-U2中256个专家的路由秘密：分组受限Top-K、Expert Bias与Fused MoE详解".
 * "The pitfalls page" is the InternLumina-U2 training-pitfalls article
 *   (m.lqnn.cn/news/279712), section "MoE 负载均衡 Loss 别忘加".
 *
 * Readings taken where the pages are silent or garbled (each one is listed
 * with its reason in the design notes of the repository):
 *   - group scores and the final top-k both use the biased score s + bias;
 *     the weights use the unbiased s (routing page, section 三);
 *   - ties go to the lower index, for groups and for experts; the k chosen
 *     experts are returned in order of (biased score desc, index asc);
 *   - the normaliser is (sum of the k chosen s, in that order, in fp32) + eps,
 *     then w = fp32(fp32(s / den) * rsf)  (routing page, section 二 step 3);
 *   - the SwiGLU intermediate silu(G) * U is rounded to bf16 once, because it
 *     is the bf16 operand of the down projection;
 *   - the shared expert is added unscaled (routing page, section 五).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fused
 * multiply-add contraction, so x86 and Arm give identical results).
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int T, H, E, n_group, topk_group, k, I, Is;
    float rsf, eps;
} orc_cfg;

/* Thread count of the OpenMP loops below (the CPU baseline reports it). */
void orc_set_threads(int n)
{
    if (n > 0)
        omp_set_num_threads(n);
}

int orc_max_threads(void)
{
    return omp_get_max_threads();
}

/* ---------------------------------------------------------------- bf16 */

/* bf16 is the top half of an IEEE binary32. */
double orc_bf16_value(uint16_t v)
{
    uint32_t u = (uint32_t)v << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* binary32 -> bf16, round to nearest, ties to even; NaN stays a quiet NaN. */
uint16_t orc_bf16_round(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

void orc_bf16_round_array(const float *in, uint16_t *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = orc_bf16_round(in[i]);
}

/* ------------------------------------------------------ routing page 二.1 */

/* Router linear layer in fp32 (routing page, section 二, step 1):
 * logits[t, e] = sum_h x[t, h] * W[e, h].  Here every product and the sum are
 * exact to double precision and the result is rounded once to fp32. */
void orc_router_logits(int T, int H, int E, const uint16_t *x, const float *W, float *logits)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const uint16_t *xt = x + (size_t)t * H;
        for (int e = 0; e < E; ++e) {
            const float *we = W + (size_t)e * H;
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += orc_bf16_value(xt[h]) * (double)we[h];
            logits[(size_t)t * E + e] = (float)acc;
        }
    }
}

/* Sigmoid scoring (routing page, section 二, step 1): each expert is scored
 * on its own, s = 1 / (1 + exp(-logit)), computed in double, rounded to fp32. */
static float sigmoid_f32(float logit)
{
    return (float)(1.0 / (1.0 + exp(-(double)logit)));
}

/* (value desc, index asc) */
static int before(float va, int ia, float vb, int ib)
{
    return va > vb || (va == vb && ia < ib);
}

/* Group-limited top-k for every token, from fp32 logits.
 *
 * Routing page, section 二 step 2: the E experts are cut in order into n_group
 * groups of E/n_group; a group's score is the sum of its two highest scores;
 * the topk_group best groups survive and the others are masked to -inf; the
 * top k of the surviving experts are chosen.  Section 三: the score used for
 * choosing is s + expert_bias.  Section 二 step 3: the weights are the
 * unbiased s of the chosen experts, divided by (their sum + eps), times rsf.
 *
 * Outputs: idx [T,k], w [T,k]; optional scores [T,E] (the unbiased s);
 * optional margins [T] in double: the gap between the topk_group-th and the
 * next group score, and between the k-th and the next surviving biased score
 * (+inf where there is no next one).
 *
 * Returns 0, or -1 for an unsupported shape, -2 for a non-finite input.
 */
int orc_route(const orc_cfg *c, const float *logits, const float *bias,
              int32_t *idx, float *w, float *scores,
              double *margin_group, double *margin_expert)
{
    const int E = c->E, G = c->n_group, TG = c->topk_group, K = c->k;
    if (G <= 0 || E % G != 0 || E / G < 2 || TG < 1 || TG > G || K < 1 || K > TG * (E / G))
        return -1;
    const int GS = E / G;
    int bad = 0;

#pragma omp parallel
    {
        float *s = malloc(sizeof(float) * E);
        float *b = malloc(sizeof(float) * E);
        float *g = malloc(sizeof(float) * G);
        int *gorder = malloc(sizeof(int) * G);
        int *cand = malloc(sizeof(int) * E);
#pragma omp for schedule(static)
        for (int t = 0; t < c->T; ++t) {
            const float *L = logits + (size_t)t * E;
            for (int e = 0; e < E; ++e) {
                if (!isfinite(L[e]) || (bias && !isfinite(bias[e]))) {
#pragma omp atomic write
                    bad = 1;
                }
                s[e] = sigmoid_f32(L[e]);
                b[e] = s[e] + (bias ? bias[e] : 0.0f); /* one fp32 add */
                if (scores)
                    scores[(size_t)t * E + e] = s[e];
            }
            /* group score = top-1 + top-2 of the biased scores in the group */
            for (int j = 0; j < G; ++j) {
                float m1 = -INFINITY, m2 = -INFINITY;
                for (int q = 0; q < GS; ++q) {
                    float v = b[j * GS + q];
                    if (v > m1) {
                        m2 = m1;
                        m1 = v;
                    } else if (v > m2) {
                        m2 = v;
                    }
                }
                g[j] = m1 + m2;
            }
            /* order the groups by (score desc, index asc): selection sort */
            for (int j = 0; j < G; ++j)
                gorder[j] = j;
            for (int a = 0; a < G; ++a)
                for (int z = a + 1; z < G; ++z)
                    if (before(g[gorder[z]], gorder[z], g[gorder[a]], gorder[a])) {
                        int tmp = gorder[a];
                        gorder[a] = gorder[z];
                        gorder[z] = tmp;
                    }
            if (margin_group)
                margin_group[t] = (TG < G) ? (double)g[gorder[TG - 1]] - (double)g[gorder[TG]] : INFINITY;
            /* survivors: the experts of the kept groups (the rest are -inf) */
            int nc = 0;
            for (int a = 0; a < TG; ++a)
                for (int q = 0; q < GS; ++q)
                    cand[nc++] = gorder[a] * GS + q;
            /* partial selection sort of the survivors by (b desc, index asc) */
            for (int a = 0; a < K && a < nc; ++a)
                for (int z = a + 1; z < nc; ++z)
                    if (before(b[cand[z]], cand[z], b[cand[a]], cand[a])) {
                        int tmp = cand[a];
                        cand[a] = cand[z];
                        cand[z] = tmp;
                    }
            if (margin_expert) {
                if (K < nc) {
                    /* best remaining survivor after the first K */
                    int best = cand[K];
                    for (int z = K + 1; z < nc; ++z)
                        if (before(b[cand[z]], cand[z], b[best], best))
                            best = cand[z];
                    margin_expert[t] = (double)b[cand[K - 1]] - (double)b[best];
                } else {
                    margin_expert[t] = INFINITY;
                }
            }
            /* weights from the unbiased scores, normalised, scaled */
            float den = 0.0f;
            for (int a = 0; a < K; ++a)
                den += s[cand[a]];
            den += c->eps;
            for (int a = 0; a < K; ++a) {
                float q = s[cand[a]] / den;
                idx[(size_t)t * K + a] = cand[a];
                w[(size_t)t * K + a] = q * c->rsf;
            }
        }
        free(s);
        free(b);
        free(g);
        free(gorder);
        free(cand);
    }
    return bad ? -2 : 0;
}

/* ---------------------------------------------- pitfalls page, aux loss */

/* Expert hit counts (routing page, section 六: a bincount of the chosen
 * indices) and the load-balancing loss E * sum_i f_i * P_i (pitfalls page):
 *   f_i = counts_i / (k T)                      (share of the k T selections)
 *   P_i = (1/T) sum_t s[t,i] / sum_e s[t,e]     (mean normalised router score)
 * P and the loss in double.  Returns the loss. */
double orc_counts_aux(int T, int E, int K, const int32_t *idx, const float *scores,
                      int32_t *counts, double *P)
{
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (long q = 0; q < (long)T * K; ++q)
        if (idx[q] >= 0 && idx[q] < E)
            counts[idx[q]] += 1;
    if (!scores || !P)
        return 0.0;
    for (int e = 0; e < E; ++e)
        P[e] = 0.0;
    for (int t = 0; t < T; ++t) {
        double tot = 0.0;
        for (int e = 0; e < E; ++e)
            tot += (double)scores[(size_t)t * E + e];
        for (int e = 0; e < E; ++e)
            P[e] += (double)scores[(size_t)t * E + e] / tot;
    }
    double aux = 0.0;
    for (int e = 0; e < E; ++e) {
        P[e] /= (double)T;
        aux += ((double)counts[e] / ((double)K * T)) * P[e];
    }
    return (double)E * aux;
}

/* --------------------------------------------- routing page 四 and 五 */

/* One SwiGLU expert on one token (routing page, section 四: gate, up and down
 * stacked as [experts, 512, 2048]):
 *   G_i = x . Wgu[i, :],  U_i = x . Wgu[I + i, :]     (i < I)
 *   a_i = bf16(fp32(silu(G_i) * U_i)),  silu(z) = z / (1 + exp(-z))
 *   y_h = sum_i a_i * Wd[i, h]
 * and y * weight is added to acc.  Wgu is [2I, H] (gate rows, then up rows),
 * Wd is [I, H]; all products and sums in double. */
static void swiglu_expert_add(int H, int I, const double *x, const uint16_t *Wgu,
                              const uint16_t *Wd, double weight, double *a, double *acc, int round_act)
{
    for (int i = 0; i < I; ++i) {
        const uint16_t *wg = Wgu + (size_t)i * H;
        const uint16_t *wu = Wgu + (size_t)(I + i) * H;
        double G = 0.0, U = 0.0;
        for (int h = 0; h < H; ++h) {
            G += x[h] * orc_bf16_value(wg[h]);
            U += x[h] * orc_bf16_value(wu[h]);
        }
        double act = G / (1.0 + exp(-G)) * U;
        a[i] = round_act ? orc_bf16_value(orc_bf16_round((float)act)) : act;
    }
    for (int i = 0; i < I; ++i) {
        const uint16_t *wd = Wd + (size_t)i * H;
        double ai = a[i] * weight;
        if (a[i] == 0.0)
            continue;
        for (int h = 0; h < H; ++h)
            acc[h] += ai * orc_bf16_value(wd[h]);
    }
}

/* Layer output for a list of tokens (routing page, sections 四 and 五):
 *   out[t] = sum_j w[t,j] * expert_{idx[t,j]}(x[t]) + shared(x[t]) (+ residual[t])
 * in double.  tokens (nullable) lists which rows of x to compute; out has one
 * row of H per listed token.  Indices outside [0, E) contribute nothing and
 * are reported by returning -1. */
int orc_experts_opt(const orc_cfg *c, const uint16_t *x, const uint16_t *Wgu, const uint16_t *Wd,
                    const uint16_t *sgu, const uint16_t *sd, const int32_t *idx, const float *w,
                    const uint16_t *residual, int n_tok, const int32_t *tokens, double *out, int round_act);

int orc_experts(const orc_cfg *c, const uint16_t *x, const uint16_t *Wgu, const uint16_t *Wd,
                const uint16_t *sgu, const uint16_t *sd, const int32_t *idx, const float *w,
                const uint16_t *residual, int n_tok, const int32_t *tokens, double *out)
{
    return orc_experts_opt(c, x, Wgu, Wd, sgu, sd, idx, w, residual, n_tok, tokens, out, 1);
}

/* As orc_experts; round_act = 0 keeps the SwiGLU intermediate unrounded (the
 * smooth function the backward's finite-difference checks differentiate). */
int orc_experts_opt(const orc_cfg *c, const uint16_t *x, const uint16_t *Wgu, const uint16_t *Wd,
                    const uint16_t *sgu, const uint16_t *sd, const int32_t *idx, const float *w,
                    const uint16_t *residual, int n_tok, const int32_t *tokens, double *out, int round_act)
{
    const int H = c->H, I = c->I, Is = c->Is, K = c->k, E = c->E;
    int bad = 0;
#pragma omp parallel
    {
        double *xd = malloc(sizeof(double) * H);
        double *a = malloc(sizeof(double) * (I > Is ? I : Is));
#pragma omp for schedule(dynamic, 1)
        for (int q = 0; q < n_tok; ++q) {
            int t = tokens ? tokens[q] : q;
            double *acc = out + (size_t)q * H;
            for (int h = 0; h < H; ++h) {
                xd[h] = orc_bf16_value(x[(size_t)t * H + h]);
                acc[h] = 0.0;
            }
            for (int j = 0; j < K; ++j) {
                int e = idx[(size_t)t * K + j];
                if (e < 0 || e >= E) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                swiglu_expert_add(H, I, xd, Wgu + (size_t)e * 2 * I * H, Wd + (size_t)e * I * H,
                                  (double)w[(size_t)t * K + j], a, acc, round_act);
            }
            if (sgu && sd)
                swiglu_expert_add(H, Is, xd, sgu, sd, 1.0, a, acc, round_act);
            if (residual)
                for (int h = 0; h < H; ++h)
                    acc[h] += orc_bf16_value(residual[(size_t)t * H + h]);
        }
        free(xd);
        free(a);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------- backward of the expert stage */

/* Gradients of one SwiGLU expert applied to one row, for an output gradient
 * dy (the gradient of this expert's output row y = a . Wd):
 *   G = x . Wg^T, U = x . Wu^T, a = silu(G) * U (bf16-rounded when round_act,
 *   the rounding passed through as the identity), y = a . Wd;
 *   dWd += a (x) dy,  da = Wd . dy,
 *   dG = da * U * s * (1 + G * (1 - s)),  dU = da * G * s   (s = sigmoid(G)),
 *   dWg += dG (x) x,  dWu += dU (x) x,  dx = dG . Wg + dU . Wu.
 * Returns <dout_row, y> (scale 1/weight applied by the caller) through *ydot
 * when dout_row is not NULL.  Everything in double. */
static void swiglu_expert_backward(int H, int I, const double *x, const uint16_t *Wgu, const uint16_t *Wd,
                                   const double *dy, int round_act, double *dWgu, double *dWd, double *dx,
                                   const double *dout_row, double *ydot)
{
    double dot = 0.0;
    for (int h = 0; h < H; ++h)
        dx[h] = 0.0;
    for (int i = 0; i < I; ++i) {
        const uint16_t *wg = Wgu + (size_t)i * H;
        const uint16_t *wu = Wgu + (size_t)(I + i) * H;
        const uint16_t *wd = Wd + (size_t)i * H;
        double G = 0.0, U = 0.0;
        for (int h = 0; h < H; ++h) {
            G += x[h] * orc_bf16_value(wg[h]);
            U += x[h] * orc_bf16_value(wu[h]);
        }
        const double sg = 1.0 / (1.0 + exp(-G));
        const double act = G * sg * U;
        const double a = round_act ? orc_bf16_value(orc_bf16_round((float)act)) : act;
        double da = 0.0;
        for (int h = 0; h < H; ++h) {
            const double wdh = orc_bf16_value(wd[h]);
            da += wdh * dy[h];
            if (dout_row)
                dot += a * wdh * dout_row[h];
        }
        double *gd = dWd + (size_t)i * H;
        for (int h = 0; h < H; ++h)
            gd[h] += a * dy[h];
        const double dG = da * U * sg * (1.0 + G * (1.0 - sg));
        const double dU = da * G * sg;
        double *gg = dWgu + (size_t)i * H;
        double *gu = dWgu + (size_t)(I + i) * H;
        for (int h = 0; h < H; ++h) {
            gg[h] += dG * x[h];
            gu[h] += dU * x[h];
            dx[h] += dG * orc_bf16_value(wg[h]) + dU * orc_bf16_value(wu[h]);
        }
    }
    if (ydot)
        *ydot = dot;
}

/* Backward of orc_experts (routing fixed, residual passed straight through):
 * given dout [T, H] (double), writes
 *   dx   [T, H]      = sum_j w[t,j] * d expert_j / dx + d shared / dx,
 *   dWgu [E, 2I, H], dWd [E, I, H], dsgu [2Is, H], dsd [Is, H]  (sums over tokens),
 *   dw   [T, k]      = <dout[t], expert_{idx[t,j]}(x[t])>.
 * Each expert's gradients are summed by one thread over its tokens in token
 * order; dx[t] adds the pairs j = 0 .. k-1, then the shared expert, in order.
 * Returns -1 if an expert index is out of range (the pair is skipped). */
int orc_experts_backward(const orc_cfg *c, const uint16_t *x, const uint16_t *Wgu, const uint16_t *Wd,
                         const uint16_t *sgu, const uint16_t *sd, const int32_t *idx, const float *w,
                         const double *dout, int round_act, double *dx, double *dWgu, double *dWd,
                         double *dsgu, double *dsd, double *dw)
{
    const int T = c->T, H = c->H, I = c->I, Is = c->Is, K = c->k, E = c->E;
    int bad = 0;
    double *dxp = calloc((size_t)T * (K + 1) * H, sizeof(double));   /* per (token, pair) */
    memset(dWgu, 0, sizeof(double) * (size_t)E * 2 * I * H);
    memset(dWd, 0, sizeof(double) * (size_t)E * I * H);
    if (dsgu)
        memset(dsgu, 0, sizeof(double) * (size_t)2 * Is * H);
    if (dsd)
        memset(dsd, 0, sizeof(double) * (size_t)Is * H);
    for (size_t i = 0; i < (size_t)T * K; ++i)
        dw[i] = 0.0;
#pragma omp parallel
    {
        double *xd = malloc(sizeof(double) * H);
        double *dy = malloc(sizeof(double) * H);
#pragma omp for schedule(dynamic, 1)
        for (int e = 0; e <= E; ++e) {             /* e == E: the shared expert */
            if (e == E && !(sgu && sd))
                continue;
            for (int t = 0; t < T; ++t) {
                for (int j = 0; j <= K; ++j) {
                    double wt;
                    if (e < E) {
                        if (j == K || idx[(size_t)t * K + j] != e)
                            continue;
                        wt = (double)w[(size_t)t * K + j];
                    } else {
                        if (j != K)
                            continue;
                        wt = 1.0;
                    }
                    for (int h = 0; h < H; ++h) {
                        xd[h] = orc_bf16_value(x[(size_t)t * H + h]);
                        dy[h] = wt * dout[(size_t)t * H + h];
                    }
                    double ydot = 0.0;
                    if (e < E)
                        swiglu_expert_backward(H, I, xd, Wgu + (size_t)e * 2 * I * H, Wd + (size_t)e * I * H,
                                               dy, round_act, dWgu + (size_t)e * 2 * I * H,
                                               dWd + (size_t)e * I * H, dxp + ((size_t)t * (K + 1) + j) * H,
                                               dout + (size_t)t * H, &ydot);
                    else
                        swiglu_expert_backward(H, Is, xd, sgu, sd, dy, round_act, dsgu, dsd,
                                               dxp + ((size_t)t * (K + 1) + K) * H, NULL, NULL);
                    if (e < E)
                        dw[(size_t)t * K + j] = ydot;
                }
            }
        }
        free(xd);
        free(dy);
    }
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < K; ++j) {
            const int e = idx[(size_t)t * K + j];
            if (e < 0 || e >= E)
                bad = 1;
        }
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j <= K; ++j)
                acc += dxp[((size_t)t * (K + 1) + j) * H + h];
            dx[(size_t)t * H + h] = acc;
        }
    free(dxp);
    return bad ? -1 : 0;
}

/* ------------------------------------------------ stacking (routing page 五) */

/* Pre-norm in front of each MoE block when layers are stacked into decoder
 * layers (routing page, section 五 names the decoder layer, not its norm; the
 * reading taken is an RMS norm with unit weight):
 *   out[t, h] = bf16( x[t, h] / sqrt(mean_h x[t, h]^2 + eps) ), in double. */
void orc_rmsnorm(int T, int H, const uint16_t *x, float eps, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int h = 0; h < H; ++h) {
            double v = orc_bf16_value(x[(size_t)t * H + h]);
            ss += v * v;
        }
        double inv = 1.0 / sqrt(ss / (double)H + (double)eps);
        for (int h = 0; h < H; ++h)
            out[(size_t)t * H + h] = orc_bf16_round((float)(orc_bf16_value(x[(size_t)t * H + h]) * inv));
    }
}

/* ------------------------------------------ routing page 三 and 六 (training) */

/* Expert-bias feedback and hit tracking after a routing step.
 * Routing page, section 三: during training the bias of cold experts is
 * raised and that of overloaded experts lowered; read here as a sign step
 * around the balanced load k T / E:
 *   bias[e] = fp32( bias[e] + step ),  step = +gamma if counts[e] < k T / E,
 *                                              -gamma if counts[e] > k T / E, 0 otherwise.
 * Section 六: the running per-expert totals accumulate every step's counts.
 * Either output may be NULL. */
void orc_expert_feedback(int E, int T, int K, const int32_t *counts, float gamma, float *bias, int64_t *totals)
{
    const double mean = (double)K * (double)T / (double)E;
    for (int e = 0; e < E; ++e) {
        if (totals)
            totals[e] += counts[e];
        if (bias) {
            float step = 0.0f;
            if ((double)counts[e] < mean)
                step = gamma;
            else if ((double)counts[e] > mean)
                step = -gamma;
            bias[e] = bias[e] + step;
        }
    }
}
