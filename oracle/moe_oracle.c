/*
 * moe_oracle.c -- plain, slow CPU oracle for the forward pass of a top-k routed
 * Mixture-of-Experts SwiGLU FFN layer with optional shared experts.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Sources (pages of the subject, cited by title and section):
 *   [H]  "混合专家 MoE" (ai-infra-handbooks, Transformer 解剖), sections
 *        "结构", "实现：逐 token 与按专家分组" (listing moe.py: Expert, MoE.route,
 *        forward_naive, forward_grouped), "负载均衡" (aux_loss listing),
 *        "练习" (exercise 1 parameter count).
 *   [N]  "混合专家模型 (MoE)：大规模稀疏条件计算的架构与工程实践", section
 *        三.1 "容量因子 (Capacity Factor) 与 Token 丢弃策略" and 一.1 (shared
 *        experts always active).
 *
 * Precision.  The router is fp32 as the layer definition fixes it: each logit
 * is the fp32 rounding of the exact dot product (accumulated in fp64 from the
 * exact fp32 x fp32 products), the softmax is evaluated in fp64 and each
 * probability rounded once to fp32; top-k and the near-tie gap are decided on
 * those fp32 probabilities.  Everything in the expert FFNs is fp64; for bf16
 * layers the SwiGLU hidden vector h is rounded to bf16 before the down
 * projection (the single intermediate rounding point of the bf16 path) and the
 * output is rounded once to bf16.  bf16 inputs are widened exactly.
 *
 * Readings where the pages are silent:
 *   - top-k orders slots by probability descending, ties to the lower index;
 *   - capacity C = ceil(CF * N * k / E); an expert keeps the first C of its
 *     assignments in (token, slot) order; a dropped assignment contributes 0
 *     and the remaining weights are not renormalised; shared experts still
 *     apply to every token;
 *   - f_i = (assignments to expert i before dropping) / (N * k),
 *     P_i = mean over tokens of the router probability of expert i.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_W4 2    /* weights only: 4-bit codes + one fp32 scale per 128 inputs (orc_w4) */

/* A W4A16 weight matrix [rows, cols]: q packs two signed 4-bit codes per byte (even column in
 * the low nibble), s holds one fp32 scale per 128 consecutive columns of a row, group-major:
 * s[g * rows + r] is the scale of row r, columns [128 g, 128 g + 128). */
typedef struct {
    const uint8_t *q;
    const float *s;
    int64_t rows;
} orc_w4;

#define ORC_W4_GROUP 128

/* ---------- scalar conversions ---------- */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even (bf16: 8 significant
 * bits, 8 exponent bits, subnormal quantum 2^-133).  Returns the bf16 bits. */
uint16_t oracle_round_bf16(double v)
{
    double r;
    if (isnan(v))
        return (uint16_t)0x7FC0;
    if (v == 0.0 || isinf(v)) {
        r = v;
    } else if (fabs(v) < ldexp(1.0, -126)) {
        r = ldexp(nearbyint(ldexp(v, 133)), -133);
    } else {
        int e;
        double m = frexp(v, &e);            /* v = m * 2^e, 0.5 <= |m| < 1 */
        r = ldexp(nearbyint(ldexp(m, 8)), e - 8);
    }
    /* largest finite bf16 is (2 - 2^-7) * 2^127 */
    if (fabs(r) > ldexp(255.0, 120))
        r = copysign(INFINITY, r);
    float f = (float)r;                     /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

static double round_to_bf16_value(double v)
{
    return bf16_bits_to_double(oracle_round_bf16(v));
}

/* element i of a matrix stored as fp32 or bf16 */
static double elem(const void *p, int dtype, int64_t i)
{
    if (dtype == ORC_BF16)
        return bf16_bits_to_double(((const uint16_t *)p)[i]);
    return (double)((const float *)p)[i];
}

/* element (row, col) of a weight matrix with `cols` columns, stored fp32, bf16 or W4 */
static double wval(const void *p, int wdtype, int64_t row, int64_t col, int64_t cols)
{
    if (wdtype == ORC_W4) {
        const orc_w4 *m = (const orc_w4 *)p;
        uint8_t byte = m->q[(row * cols + col) / 2];
        int nib = (col & 1) ? (byte >> 4) : (byte & 15);
        int code = nib >= 8 ? nib - 16 : nib;                  /* two's complement, 4 bits */
        return (double)code * (double)m->s[(col / ORC_W4_GROUP) * m->rows + row];
    }
    return elem(p, wdtype, row * cols + col);
}

/* ---------- router: logits, softmax, top-k, renormalise ([H] MoE.route) ---------- */

/* For one token: probs[E] (fp32), idx[k], w[k], gap.  Returns 0. */
static void route_token(int d, int E, int k, int dtype, const void *x, int64_t t,
                        const float *W_r, const float *b_r, int bias_mode, int renorm,
                        float *probs, int32_t *idx, float *w, float *gap, double *lse)
{
    float *logit = (float *)malloc(sizeof(float) * (size_t)E);
    float *sel = (float *)malloc(sizeof(float) * (size_t)E);
    unsigned char *chosen = (unsigned char *)calloc((size_t)E, 1);

    /* logits: l[e] = (b_e if the bias enters the logits) + sum_i x[t,i] * W_r[e,i],
     * rounded once to fp32 */
    for (int e = 0; e < E; e++) {
        double acc = (b_r && bias_mode == 1) ? (double)b_r[e] : 0.0;
        for (int i = 0; i < d; i++)
            acc += elem(x, dtype, t * (int64_t)d + i) * (double)W_r[(int64_t)e * d + i];
        logit[e] = (float)acc;
    }

    /* softmax over all E experts, with the maximum subtracted */
    double mx = logit[0];
    for (int e = 1; e < E; e++)
        if (logit[e] > mx)
            mx = logit[e];
    double s = 0.0;
    for (int e = 0; e < E; e++)
        s += exp((double)logit[e] - mx);
    for (int e = 0; e < E; e++)
        probs[e] = (float)(exp((double)logit[e] - mx) / s);
    /* log-sum-exp of the raw logits (the z-loss term of "混合专家模型 (MoE)" section 三.3) */
    if (lse)
        *lse = mx + log(s);

    /* selection score: the probability, or with a selection-only bias ("混合专家 MoE",
     * 负载均衡: the bias only picks the top-k, it does not change the weights) p_e + b_e,
     * rounded once to fp32 */
    for (int e = 0; e < E; e++)
        sel[e] = (b_r && bias_mode == 2) ? (float)((double)probs[e] + (double)b_r[e]) : probs[e];

    /* top-k: k rounds of "largest score not yet chosen", ties to the lower index */
    for (int j = 0; j < k; j++) {
        int best = -1;
        for (int e = 0; e < E; e++)
            if (!chosen[e] && (best < 0 || sel[e] > sel[best]))
                best = e;
        idx[j] = best;
        chosen[best] = 1;
    }

    /* gap between the k-th and the (k+1)-th score (none when k == E) */
    if (k < E) {
        int nb = -1;
        for (int e = 0; e < E; e++)
            if (!chosen[e] && (nb < 0 || sel[e] > sel[nb]))
                nb = e;
        *gap = (float)((double)sel[idx[k - 1]] - (double)sel[nb]);
    } else {
        *gap = INFINITY;
    }

    /* renormalise the k selected weights so they sum to one */
    double ws = 0.0;
    for (int j = 0; j < k; j++)
        ws += (double)probs[idx[j]];
    for (int j = 0; j < k; j++)
        w[j] = renorm ? (float)((double)probs[idx[j]] / ws) : probs[idx[j]];

    free(logit);
    free(sel);
    free(chosen);
}

/*
 * oracle_route: router for all N tokens.
 *   x [N,d] (fp32 or bf16 bits), W_r [E,d] fp32, b_r [E] fp32 or NULL;
 *   bias_mode 1: b_r is added to the logits; 2: b_r is added to the probabilities for the
 *   top-k choice only (the weights and probs stay unbiased).
 *   idx [N,k] int32, w [N,k] fp32; probs [N,E] fp32 and gap [N] fp32 may be NULL.
 */
int oracle_route(int64_t N, int d, int E, int k, int dtype, const void *x,
                 const float *W_r, const float *b_r, int bias_mode, int renorm,
                 int32_t *idx, float *w, float *probs, float *gap, double *lse)
{
    if (N < 0 || d <= 0 || E <= 0 || k <= 0 || k > E)
        return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < N; t++) {
        float *p = (float *)malloc(sizeof(float) * (size_t)E);
        float g;
        route_token(d, E, k, dtype, x, t, W_r, b_r, bias_mode, renorm, p, idx + t * k, w + t * k, &g,
                    lse ? lse + t : NULL);
        if (probs)
            memcpy(probs + t * (int64_t)E, p, sizeof(float) * (size_t)E);
        if (gap)
            gap[t] = g;
        free(p);
    }
    return 0;
}

/* ---------- capacity ([N] 三.1) ---------- */

/* C = ceil(CF * N * k / E); -1 when CF <= 0 (no limit). */
int64_t oracle_capacity(int64_t N, int k, int E, double cf)
{
    if (!(cf > 0.0))
        return -1;
    return (int64_t)ceil(cf * (double)N * (double)k / (double)E);
}

/* ---------- grouping by expert ([H] forward_grouped: flatten, stable argsort, bincount) ---------- */

/*
 * oracle_permute: flat slot f = t*k + j goes to expert idx[f].
 *   counts[E]       = histogram of idx                       (bincount)
 *   offsets[E+1]    = exclusive prefix sum of counts         (segment starts)
 *   perm[N*k]       = slots sorted by expert, stable         (argsort(stable=True))
 *   kept[E]         = min(counts, C)
 *   kept_offsets[E+1] = exclusive prefix sum of kept
 *   pos[N*k]        = row of slot f in the compacted kept order, or -1 if dropped
 * capacity < 0 means no limit.  Returns 1 on an index outside [0, E).
 */
int oracle_permute(int64_t N, int k, int E, const int32_t *idx, int64_t capacity,
                   int32_t *counts, int32_t *offsets, int32_t *kept, int32_t *kept_offsets,
                   int32_t *perm, int32_t *pos)
{
    if (N < 0 || k <= 0 || E <= 0)
        return 1;
    int64_t A = N * k;
    for (int64_t f = 0; f < A; f++)
        if (idx[f] < 0 || idx[f] >= E)
            return 1;
    for (int e = 0; e < E; e++)
        counts[e] = 0;
    for (int64_t f = 0; f < A; f++)
        counts[idx[f]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; e++)
        offsets[e + 1] = offsets[e] + counts[e];
    kept_offsets[0] = 0;
    for (int e = 0; e < E; e++) {
        kept[e] = (capacity >= 0 && counts[e] > capacity) ? (int32_t)capacity : counts[e];
        kept_offsets[e + 1] = kept_offsets[e] + kept[e];
    }
    /* counting sort: walking f in increasing order keeps equal keys stable */
    int32_t *cursor = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t f = 0; f < A; f++) {
        int e = idx[f];
        int32_t r = cursor[e]++;
        perm[offsets[e] + r] = (int32_t)f;
        pos[f] = (r < kept[e]) ? kept_offsets[e] + r : -1;
    }
    free(cursor);
    return 0;
}

/* ---------- one expert on one token ([H] Expert.forward) ---------- */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* y[d] = W_down (silu(W_gate x) * (W_up x)); W_gate/W_up [F,d], W_down [d,F]. */
static void swiglu_expert(const double *xt, int d, int F, int dtype, const void *Wg,
                          const void *Wu, const void *Wd, int round_h, double *y)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)F);
    for (int n = 0; n < F; n++) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < d; i++) {
            g += wval(Wg, dtype, n, i, d) * xt[i];
            u += wval(Wu, dtype, n, i, d) * xt[i];
        }
        double hv = silu(g) * u;
        h[n] = round_h ? round_to_bf16_value(hv) : hv;
    }
    for (int i = 0; i < d; i++) {
        double acc = 0.0;
        for (int n = 0; n < F; n++)
            acc += wval(Wd, dtype, i, n, F) * h[n];
        y[i] = acc;
    }
    free(h);
}

static void store_row(void *out, int dtype, int64_t row, int d, const double *acc)
{
    for (int i = 0; i < d; i++) {
        if (dtype == ORC_BF16)
            ((uint16_t *)out)[row * d + i] = oracle_round_bf16(acc[i]);
        else
            ((float *)out)[row * d + i] = (float)acc[i];
    }
}

/*
 * oracle_moe_token: the layer output for one token ([H] forward_naive body):
 *   out_t = sum_{j : keep_t[j]} w_t[j] * Expert_{idx_t[j]}(x_t)  +  sum_s Shared_s(x_t)
 * The k chosen experts' matrices are passed as pointer arrays (Wg_k[j] is the
 * [F,d] gate matrix of expert idx_t[j], ...), the S shared experts likewise.
 * x_t [d] and out_t [d] are in the layer dtype.
 */
int oracle_moe_token_w(int d, int F, int k, int S, int Fs, int dtype, int wdtype, int round_h,
                       const void *x_t, const float *w_t, const int32_t *keep_t,
                       const void *const *Wg_k, const void *const *Wu_k, const void *const *Wd_k,
                       const void *const *Wsg, const void *const *Wsu, const void *const *Wsd,
                       void *out_t)
{
    double *xt = (double *)malloc(sizeof(double) * (size_t)d);
    double *acc = (double *)calloc((size_t)d, sizeof(double));
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < d; i++)
        xt[i] = elem(x_t, dtype, i);
    for (int j = 0; j < k; j++) {
        if (!keep_t[j])
            continue;
        swiglu_expert(xt, d, F, wdtype, Wg_k[j], Wu_k[j], Wd_k[j], round_h, y);
        for (int i = 0; i < d; i++)
            acc[i] += (double)w_t[j] * y[i];
    }
    for (int s = 0; s < S; s++) {
        swiglu_expert(xt, d, Fs, wdtype, Wsg[s], Wsu[s], Wsd[s], round_h, y);
        for (int i = 0; i < d; i++)
            acc[i] += y[i];
    }
    store_row(out_t, dtype, 0, d, acc);
    free(xt);
    free(acc);
    free(y);
    return 0;
}

/* oracle_moe_token_w with the weights in the activation dtype */
int oracle_moe_token(int d, int F, int k, int S, int Fs, int dtype, int round_h,
                     const void *x_t, const float *w_t, const int32_t *keep_t,
                     const void *const *Wg_k, const void *const *Wu_k, const void *const *Wd_k,
                     const void *const *Wsg, const void *const *Wsu, const void *const *Wsd,
                     void *out_t)
{
    return oracle_moe_token_w(d, F, k, S, Fs, dtype, dtype, round_h, x_t, w_t, keep_t, Wg_k, Wu_k,
                              Wd_k, Wsg, Wsu, Wsd, out_t);
}

static const void *expert_mat(const void *bank, int dtype, int64_t e, int64_t rows, int64_t cols)
{
    size_t esz = dtype == ORC_BF16 ? 2 : 4;
    return (const char *)bank + (size_t)(e * rows * cols) * esz;
}

/*
 * oracle_keep_naive: which assignments survive the capacity limit, decided the
 * per-token way: walking tokens t = 0..N-1 and slots j = 0..k-1, an assignment
 * to expert e is kept while fewer than C earlier assignments went to e.
 * keep[N*k] gets 1/0.  capacity < 0: everything kept.
 */
void oracle_keep_naive(int64_t N, int k, int E, const int32_t *idx, int64_t capacity, int32_t *keep)
{
    int64_t *seen = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    for (int64_t t = 0; t < N; t++)
        for (int j = 0; j < k; j++) {
            int e = idx[t * k + j];
            keep[t * k + j] = (capacity < 0 || seen[e] < capacity) ? 1 : 0;
            seen[e]++;
        }
    free(seen);
}

/*
 * oracle_forward_naive: the whole layer, token by token ([H] forward_naive).
 * Weights: Wg/Wu [E,F,d], Wd [E,d,F], Wsg/Wsu [S,Fs,d], Wsd [S,d,Fs] in the layer
 * dtype (fp32 or bf16 bits); W_r fp32 [E,d]; b_r fp32 [E] or NULL.
 * Optional outputs (NULL to skip): idx/w/keep [N,k], probs [N,E], gap [N].
 */
int oracle_forward_naive(int64_t N, int d, int F, int E, int k, int S, int Fs, int dtype,
                         double cf, int renorm, int round_h,
                         const void *x, const float *W_r, const float *b_r, int bias_mode,
                         const void *Wg, const void *Wu, const void *Wd,
                         const void *Wsg, const void *Wsu, const void *Wsd,
                         void *out, int32_t *idx_o, float *w_o, int32_t *keep_o,
                         float *probs_o, float *gap_o)
{
    if (N < 0 || k > E || k <= 0 || k > 64 || S < 0 || S > 64)
        return 1;
    int64_t A = N * k;
    int32_t *idx = idx_o ? idx_o : (int32_t *)malloc(sizeof(int32_t) * (size_t)(A ? A : 1));
    float *w = w_o ? w_o : (float *)malloc(sizeof(float) * (size_t)(A ? A : 1));
    int32_t *keep = keep_o ? keep_o : (int32_t *)malloc(sizeof(int32_t) * (size_t)(A ? A : 1));
    int rc = oracle_route(N, d, E, k, dtype, x, W_r, b_r, bias_mode, renorm, idx, w, probs_o, gap_o,
                          NULL);
    if (rc) {
        if (!idx_o) free(idx);
        if (!w_o) free(w);
        if (!keep_o) free(keep);
        return rc;
    }
    oracle_keep_naive(N, k, E, idx, oracle_capacity(N, k, E, cf), keep);
    size_t esz = dtype == ORC_BF16 ? 2 : 4;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < N; t++) {
        const void *gk[64], *uk[64], *dk[64], *sg[64], *su[64], *sd[64];
        for (int j = 0; j < k; j++) {
            int e = idx[t * k + j];
            gk[j] = expert_mat(Wg, dtype, e, F, d);
            uk[j] = expert_mat(Wu, dtype, e, F, d);
            dk[j] = expert_mat(Wd, dtype, e, d, F);
        }
        for (int s = 0; s < S; s++) {
            sg[s] = expert_mat(Wsg, dtype, s, Fs, d);
            su[s] = expert_mat(Wsu, dtype, s, Fs, d);
            sd[s] = expert_mat(Wsd, dtype, s, d, Fs);
        }
        oracle_moe_token(d, F, k, S, Fs, dtype, round_h, (const char *)x + (size_t)(t * d) * esz,
                         w + t * k, keep + t * k, gk, uk, dk, sg, su, sd,
                         (char *)out + (size_t)(t * d) * esz);
    }
    if (!idx_o) free(idx);
    if (!w_o) free(w);
    if (!keep_o) free(keep);
    return 0;
}

/*
 * oracle_forward_grouped: the same layer organised per expert ([H]
 * forward_grouped): route, stable-sort the slots by expert, then for each
 * expert run its kept tokens and add w * y back at the token's row; shared
 * experts on every token last.  Used to check that both organisations agree.
 */
int oracle_forward_grouped(int64_t N, int d, int F, int E, int k, int S, int Fs, int dtype,
                           double cf, int renorm, int round_h,
                           const void *x, const float *W_r, const float *b_r, int bias_mode,
                           const void *Wg, const void *Wu, const void *Wd,
                           const void *Wsg, const void *Wsu, const void *Wsd, void *out)
{
    if (N < 0 || k > E || k <= 0)
        return 1;
    int64_t A = N * k;
    size_t a1 = (size_t)(A ? A : 1);
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * a1);
    float *w = (float *)malloc(sizeof(float) * a1);
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * a1);
    int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * a1);
    int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int32_t *kept = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int32_t *kept_off = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    double *acc = (double *)calloc((size_t)(N * d ? N * d : 1), sizeof(double));
    double *xt = (double *)malloc(sizeof(double) * (size_t)d);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    int rc = oracle_route(N, d, E, k, dtype, x, W_r, b_r, bias_mode, renorm, idx, w, NULL, NULL,
                          NULL);
    if (!rc)
        rc = oracle_permute(N, k, E, idx, oracle_capacity(N, k, E, cf), counts, offsets, kept,
                            kept_off, perm, pos);
    if (!rc) {
        for (int e = 0; e < E; e++) {
            for (int32_t r = 0; r < kept[e]; r++) {       /* empty experts are skipped */
                int32_t f = perm[offsets[e] + r];
                int64_t t = f / k;
                for (int i = 0; i < d; i++)
                    xt[i] = elem(x, dtype, t * d + i);
                swiglu_expert(xt, d, F, dtype, expert_mat(Wg, dtype, e, F, d),
                              expert_mat(Wu, dtype, e, F, d), expert_mat(Wd, dtype, e, d, F),
                              round_h, y);
                for (int i = 0; i < d; i++)
                    acc[t * d + i] += (double)w[f] * y[i];
            }
        }
        for (int s = 0; s < S; s++)
            for (int64_t t = 0; t < N; t++) {
                for (int i = 0; i < d; i++)
                    xt[i] = elem(x, dtype, t * d + i);
                swiglu_expert(xt, d, Fs, dtype, expert_mat(Wsg, dtype, s, Fs, d),
                              expert_mat(Wsu, dtype, s, Fs, d), expert_mat(Wsd, dtype, s, d, Fs),
                              round_h, y);
                for (int i = 0; i < d; i++)
                    acc[t * d + i] += y[i];
            }
        for (int64_t t = 0; t < N; t++)
            store_row(out, dtype, t, d, acc + t * d);
    }
    free(idx); free(w); free(perm); free(pos); free(counts); free(kept);
    free(offsets); free(kept_off); free(acc); free(xt); free(y);
    return rc;
}

/* ---------- load-balance statistics ([H] 负载均衡, aux_loss) ---------- */

/*
 * oracle_stats:
 *   f[e] = #{slots routed to e, before dropping} / (N*k)
 *   P[e] = (1/N) sum_t probs[t,e]
 *   aux  = E * sum_e f[e] * P[e]
 *   counters[0] = dropped assignments, [1] = tokens with every assignment dropped,
 *   counters[2] = tokens whose k-th and (k+1)-th probabilities differ by < tie_eps.
 * keep [N*k] (NULL = all kept), gap [N] (NULL = no tie count).
 */
int oracle_stats(int64_t N, int E, int k, const int32_t *idx, const float *probs,
                 const int32_t *keep, const float *gap, double tie_eps,
                 double *f, double *P, double *aux, int64_t *counters)
{
    if (N <= 0 || E <= 0 || k <= 0)
        return 1;
    for (int e = 0; e < E; e++) {
        f[e] = 0.0;
        P[e] = 0.0;
    }
    for (int64_t s = 0; s < N * k; s++) {
        if (idx[s] < 0 || idx[s] >= E)
            return 1;
        f[idx[s]] += 1.0;
    }
    for (int e = 0; e < E; e++)
        f[e] /= (double)(N * k);
    for (int e = 0; e < E; e++) {
        double s = 0.0;
        for (int64_t t = 0; t < N; t++)
            s += (double)probs[t * E + e];
        P[e] = s / (double)N;
    }
    double a = 0.0;
    for (int e = 0; e < E; e++)
        a += f[e] * P[e];
    *aux = (double)E * a;
    counters[0] = counters[1] = counters[2] = 0;
    for (int64_t t = 0; t < N; t++) {
        int any = 0;
        for (int j = 0; j < k; j++) {
            int kp = keep ? keep[t * k + j] : 1;
            if (!kp)
                counters[0]++;
            any |= kp;
        }
        if (!any)
            counters[1]++;
        if (gap && (double)gap[t] < tie_eps)
            counters[2]++;
    }
    return 0;
}

/* ---------- backward pass (chain rule through the forward above) ---------- */

/*
 * One SwiGLU expert's backward for one token: the forward h = silu(W_g x) * (W_u x) (rounded to
 * bf16 when round_h, the forward's rounding point, whose derivative is taken as 1),
 * y = W_d h; the upstream gradient of y is wgt * dout.  Accumulates dW_g += dg x^T,
 * dW_u += du x^T, dW_d += dy h^T and dx += W_g^T dg + W_u^T du; returns <dout, y>.
 */
static double swiglu_backward(const double *xt, int d, int F, int wdtype, const void *Wg,
                              const void *Wu, const void *Wd, int round_h, double wgt,
                              const double *dout, double *dx, double *dWg, double *dWu,
                              double *dWd)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)F);
    double *u = (double *)malloc(sizeof(double) * (size_t)F);
    double *h = (double *)malloc(sizeof(double) * (size_t)F);
    double *dh = (double *)malloc(sizeof(double) * (size_t)F);
    for (int n = 0; n < F; n++) {
        double gv = 0.0, uv = 0.0;
        for (int i = 0; i < d; i++) {
            gv += wval(Wg, wdtype, n, i, d) * xt[i];
            uv += wval(Wu, wdtype, n, i, d) * xt[i];
        }
        g[n] = gv;
        u[n] = uv;
        double hv = silu(gv) * uv;
        h[n] = round_h ? round_to_bf16_value(hv) : hv;
    }
    /* y = W_d h, <dout, y>, dh = W_d^T dy, dW_d += dy h^T with dy = wgt * dout */
    double dot = 0.0;
    for (int n = 0; n < F; n++)
        dh[n] = 0.0;
    for (int i = 0; i < d; i++) {
        double y = 0.0;
        for (int n = 0; n < F; n++)
            y += wval(Wd, wdtype, i, n, F) * h[n];
        dot += dout[i] * y;
        double dy = wgt * dout[i];
        for (int n = 0; n < F; n++) {
            dh[n] += wval(Wd, wdtype, i, n, F) * dy;
            dWd[(int64_t)i * F + n] += dy * h[n];
        }
    }
    /* h = silu(g) u: dg = dh u silu'(g), du = dh silu(g); silu'(z) = s (1 + z (1 - s)) */
    for (int n = 0; n < F; n++) {
        double sg = 1.0 / (1.0 + exp(-g[n]));
        double dg = dh[n] * u[n] * sg * (1.0 + g[n] * (1.0 - sg));
        double du = dh[n] * g[n] * sg;
        for (int i = 0; i < d; i++) {
            dWg[(int64_t)n * d + i] += dg * xt[i];
            dWu[(int64_t)n * d + i] += du * xt[i];
            dx[i] += wval(Wg, wdtype, n, i, d) * dg + wval(Wu, wdtype, n, i, d) * du;
        }
    }
    free(g);
    free(u);
    free(h);
    free(dh);
    return dot;
}

/*
 * oracle_backward: gradients of
 *     L = sum_t <dout_t, out_t> + aux_coef * L_aux + z_coef * L_z
 * with respect to x, W_r, b_r (bias_mode 1), the routed and the shared expert weights, where
 * out is the layer of oracle_forward_naive, L_aux = E sum_e f_e P_e ("混合专家 MoE", 负载均衡)
 * and L_z = (1/N) sum_t lse_t^2 (oracle_router_stats).  Readings: the top-k choice and the
 * capacity drop are piecewise constant (no gradient through the selection itself); f_e is a
 * count (constant); the bf16 rounding of h passes the gradient unchanged; the selection-only
 * bias (bias_mode 2) gets no gradient.  The routing weight w_j = p_ij / sum_sel p (renorm) so
 * dp_ij = (dw_j - sum_j' w_j' dw_j') / sum_sel p, with dw_j = <dout_t, y_j> for kept slots;
 * softmax: dl_e = p_e (dp_e - sum_e' p_e' dp_e'); the z-loss adds (2 z_coef / N) lse_t p_e.
 * All outputs fp64, zeroed first; db may be NULL.  Sequential (deterministic).
 */
int oracle_backward(int64_t N, int d, int F, int E, int k, int S, int Fs, int dtype, double cf,
                    int renorm, int round_h, const void *x, const float *W_r, const float *b_r,
                    int bias_mode, const void *Wg, const void *Wu, const void *Wd,
                    const void *Wsg, const void *Wsu, const void *Wsd, const double *dout,
                    double aux_coef, double z_coef, double *dx, double *dW_r, double *db,
                    double *dWg, double *dWu, double *dWd, double *dWsg, double *dWsu,
                    double *dWsd)
{
    if (N < 0 || k > E || k <= 0 || k > 64 || S < 0 || S > 64 || d <= 0 || F <= 0)
        return 1;
    int64_t A = N * k;
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(A ? A : 1));
    float *w = (float *)malloc(sizeof(float) * (size_t)(A ? A : 1));
    int32_t *keep = (int32_t *)malloc(sizeof(int32_t) * (size_t)(A ? A : 1));
    float *probs = (float *)malloc(sizeof(float) * (size_t)(N ? N : 1) * (size_t)E);
    double *lse = (double *)malloc(sizeof(double) * (size_t)(N ? N : 1));
    double *counts = (double *)calloc((size_t)E, sizeof(double));
    int rc = oracle_route(N, d, E, k, dtype, x, W_r, b_r, bias_mode, renorm, idx, w, probs, NULL,
                          lse);
    if (!rc) {
        oracle_keep_naive(N, k, E, idx, oracle_capacity(N, k, E, cf), keep);
        for (int64_t f = 0; f < A; f++)
            counts[idx[f]] += 1.0;
        memset(dx, 0, sizeof(double) * (size_t)N * (size_t)d);
        memset(dW_r, 0, sizeof(double) * (size_t)E * (size_t)d);
        if (db)
            memset(db, 0, sizeof(double) * (size_t)E);
        memset(dWg, 0, sizeof(double) * (size_t)E * (size_t)F * (size_t)d);
        memset(dWu, 0, sizeof(double) * (size_t)E * (size_t)F * (size_t)d);
        memset(dWd, 0, sizeof(double) * (size_t)E * (size_t)d * (size_t)F);
        if (S > 0) {
            memset(dWsg, 0, sizeof(double) * (size_t)S * (size_t)Fs * (size_t)d);
            memset(dWsu, 0, sizeof(double) * (size_t)S * (size_t)Fs * (size_t)d);
            memset(dWsd, 0, sizeof(double) * (size_t)S * (size_t)d * (size_t)Fs);
        }
        double *xt = (double *)malloc(sizeof(double) * (size_t)d);
        double *dp = (double *)malloc(sizeof(double) * (size_t)E);
        double dw[64];
        for (int64_t t = 0; t < N; t++) {
            const double *dt = dout + t * (int64_t)d;
            double *dxt = dx + t * (int64_t)d;
            for (int i = 0; i < d; i++)
                xt[i] = elem(x, dtype, t * (int64_t)d + i);
            /* routed experts */
            for (int j = 0; j < k; j++) {
                dw[j] = 0.0;
                if (!keep[t * k + j])
                    continue;
                int e = idx[t * k + j];
                dw[j] = swiglu_backward(xt, d, F, dtype, expert_mat(Wg, dtype, e, F, d),
                                        expert_mat(Wu, dtype, e, F, d),
                                        expert_mat(Wd, dtype, e, d, F), round_h,
                                        (double)w[t * k + j], dt, dxt,
                                        dWg + (int64_t)e * F * d, dWu + (int64_t)e * F * d,
                                        dWd + (int64_t)e * d * F);
            }
            /* shared experts, weight 1 */
            for (int sh = 0; sh < S; sh++)
                swiglu_backward(xt, d, Fs, dtype, expert_mat(Wsg, dtype, sh, Fs, d),
                                expert_mat(Wsu, dtype, sh, Fs, d),
                                expert_mat(Wsd, dtype, sh, d, Fs), round_h, 1.0, dt, dxt,
                                dWsg + (int64_t)sh * Fs * d, dWsu + (int64_t)sh * Fs * d,
                                dWsd + (int64_t)sh * d * Fs);
            /* routing weights -> probabilities */
            const float *pt = probs + t * (int64_t)E;
            for (int e = 0; e < E; e++)
                dp[e] = aux_coef * (double)E * (counts[e] / (double)A) / (double)N;
            double ssel = 0.0, wdw = 0.0;
            for (int j = 0; j < k; j++) {
                ssel += (double)pt[idx[t * k + j]];
                wdw += (double)w[t * k + j] * dw[j];
            }
            for (int j = 0; j < k; j++)
                dp[idx[t * k + j]] += renorm ? (dw[j] - wdw) / ssel : dw[j];
            /* softmax -> logits, plus the z-loss term */
            double pdp = 0.0;
            for (int e = 0; e < E; e++)
                pdp += (double)pt[e] * dp[e];
            for (int e = 0; e < E; e++) {
                double dl = (double)pt[e] * (dp[e] - pdp) +
                            2.0 * z_coef / (double)N * lse[t] * (double)pt[e];
                for (int i = 0; i < d; i++) {
                    dW_r[(int64_t)e * d + i] += dl * xt[i];
                    dxt[i] += dl * (double)W_r[(int64_t)e * d + i];
                }
                if (db && b_r && bias_mode == 1)
                    db[e] += dl;
            }
        }
        free(xt);
        free(dp);
    }
    free(idx);
    free(w);
    free(keep);
    free(probs);
    free(lse);
    free(counts);
    return rc;
}

/* ---------- router statistics: z-loss and importance ("混合专家模型 (MoE)", 二.2 and 三.3) ---------- */

/*
 * oracle_router_stats, plain definitions (the pages' formulas are lost; the readings):
 *   z_loss = (1/N) sum_t lse_t^2, lse_t = log sum_e exp(l_t,e) of the raw logits, before top-k;
 *   imp[e] = sum_t sum_j w_t,j [idx_t,j == e]: the gate weight each expert was assigned (the
 *            renormalised top-k weights), over every assignment before any capacity drop;
 *   cv2    = Var(imp) / Mean(imp)^2 over the E experts, population variance (0 if the mean is 0).
 * Returns 1 on bad sizes.
 */
int oracle_router_stats(int64_t N, int E, int k, const int32_t *idx, const float *w,
                        const double *lse, double *z_loss, double *imp, double *cv2)
{
    if (N < 0 || E <= 0 || k <= 0)
        return 1;
    double z = 0.0;
    for (int64_t t = 0; t < N; t++)
        z += lse[t] * lse[t];
    *z_loss = N > 0 ? z / (double)N : 0.0;
    for (int e = 0; e < E; e++)
        imp[e] = 0.0;
    for (int64_t f = 0; f < N * (int64_t)k; f++) {
        if (idx[f] < 0 || idx[f] >= E)
            return 1;
        imp[idx[f]] += (double)w[f];
    }
    double mean = 0.0;
    for (int e = 0; e < E; e++)
        mean += imp[e];
    mean /= (double)E;
    double var = 0.0;
    for (int e = 0; e < E; e++)
        var += (imp[e] - mean) * (imp[e] - mean);
    var /= (double)E;
    *cv2 = mean > 0.0 ? var / (mean * mean) : 0.0;
    return 0;
}

/* ---------- W4A16 weights ([N] 五.1: INT4 weights, BF16 activations, dequantise then compute) ---------- */

/*
 * oracle_quantize_w4: W [rows, cols] bf16 bits -> q [rows, cols/2] packed codes, s [cols/128, rows].
 * Per group of 128 consecutive columns: s = max|w| / 7 (fp32), code = w / s rounded to the nearest
 * integer (ties to even, fp32 division), clamped to [-8, 7]; an all-zero group has s = 0 and codes 0.
 * cols must be a multiple of 128.  Returns 1 on bad sizes.
 */
int oracle_quantize_w4(const uint16_t *W, int64_t rows, int cols, uint8_t *q, float *s)
{
    if (rows < 0 || cols <= 0 || cols % ORC_W4_GROUP)
        return 1;
    const int groups = cols / ORC_W4_GROUP;
    for (int64_t r = 0; r < rows; r++)
        for (int g = 0; g < groups; g++) {
            float mx = 0.0f;
            for (int c = 0; c < ORC_W4_GROUP; c++) {
                float v = (float)bf16_bits_to_double(W[r * cols + g * ORC_W4_GROUP + c]);
                if (fabsf(v) > mx)
                    mx = fabsf(v);
            }
            float sc = mx / 7.0f;
            s[(int64_t)g * rows + r] = sc;
            for (int c = 0; c < ORC_W4_GROUP; c++) {
                int64_t col = (int64_t)g * ORC_W4_GROUP + c;
                float v = (float)bf16_bits_to_double(W[r * cols + col]);
                int code = 0;
                if (sc > 0.0f) {
                    float t = nearbyintf(v / sc);
                    code = t < -8.0f ? -8 : (t > 7.0f ? 7 : (int)t);
                }
                uint8_t nib = (uint8_t)(code & 15);
                uint8_t *byte = &q[(r * cols + col) / 2];
                if (col & 1)
                    *byte = (uint8_t)((*byte & 0x0F) | (nib << 4));
                else
                    *byte = (uint8_t)((*byte & 0xF0) | nib);
            }
        }
    return 0;
}

/* oracle_dequantize_w4: W[r, c] = code * s, exact, in fp64. */
void oracle_dequantize_w4(const uint8_t *q, const float *s, int64_t rows, int cols, double *W)
{
    orc_w4 m = {q, s, rows};
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++)
            W[r * cols + c] = wval(&m, ORC_W4, r, c, cols);
}
