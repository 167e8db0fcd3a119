/*
 * specverify_oracle.c -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * A plain, slow, CPU reference of the speculative-sampling verify step in
 * IEEE double precision (sums Neumaier-compensated). Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark may load it.
 * It shares no code, header, table or constant generator with the CUDA
 * library, and it never calls it.
 *
 * What it follows (page title, then section / equation / algorithm):
 *  [DS]  "DistillSpec: Improving Speculative Decoding via Knowledge
 *        Distillation" (Zhou et al., ICLR 2024): Sec. 3 "Speculative
 *        sampling"; App. A.3, Algorithm A.1 "Speculative decoding step";
 *        App. B.3 (one temperature for target and draft).
 *  [LKM] "How speculative decoding lets a small model draft and a large one
 *        check" (explainer of Leviathan, Kalman & Matias): the quoted
 *        rule n = min({i-1 : r_i > p_i(x)/q_i(x)} U {gamma}) and the
 *        "at least one, at most gamma+1 tokens" property.
 *  [KAD] "Speculative Decoding and Distillation" (Kadimisetty notes):
 *        Part 1 steps 1-5, Part 1 "Speedup math", Part 2 temperature
 *        softmax, "Greedy vs sampling" (greedy acceptance = exact match).
 *  [SAL] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *        1, 2, 3", SC'11 -- the Philox4x32-10 counter-based generator.
 *  [DSL] "DistillSpec", Sec. 4 "DistillSpec with lossy SD" (lenience
 *        functions f_lin, f_sq, f_exp) and Algorithm A.1's rejection
 *        threshold f(p_i(y), eps) / q_i(y).
 *  [DSB] "DistillSpec", Sec. 3 (acceptance rate beta = sum min(p, q)) and
 *        Sec. 4 / App. A.1 (total variation distance as its proxy).
 *  [DIS] "Dynamic Speculation Lookahead ..." (DISCO), Sec. 3 Eq. 2 and
 *        App. D.1: the classifier's inputs are the top-k probabilities and
 *        the entropy of the draft distribution.
 *  [KGS] "Speculative Decoding and Distillation" (Kadimisetty notes),
 *        "Greedy vs sampling": sampling variants (temperature, top-k,
 *        top-p) apply to target and draft alike; the accept/resample rule
 *        then runs on the restricted distributions.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *  - uniforms: U24(x) = (2*(x>>9)+1) * 2^-24 for the accept test and
 *    U52(x0,x1) = (2*k+1) * 2^-53, k = (x0<<20)|(x1>>12), for the final
 *    draw; both are exact dyadic numbers strictly inside (0,1);
 *  - counter = (sequence b, 1-based position i, purpose, 0) with purpose 0
 *    for the accept test and 1 for the final draw; key = (seed lo, seed hi);
 *  - ties r_i == ratio_i accept (both pages reject only on a strict ">");
 *  - the final draw is the inverse CDF in index order: the smallest k with
 *    C_k > u*R, where C_k sums the weights of tokens 0..k and R is their total;
 *  - residual weights use p*max(0, -expm1(log q - log p)), which equals
 *    max(0, p-q) and does not cancel when p and q are both near one;
 *  - a residual of zero total mass (possible only through rounding) draws
 *    from p_{n+1} and is reported in draw_fallback;
 *  - a NaN or +inf logit, or a row with every logit -inf, is a bad input;
 *  - lenience: kind 0 is the lossless f(p) = p, kinds 1, 2, 3 are f_lin,
 *    f_sq and f_exp with one eps in (0, 1] per call; the residual after a
 *    rejection stays norm(max(0, p - q)) whatever the lenience;
 *  - TVD(p, q) = 1/2 sum |p - q| (only with the 1/2 does 1 - TVD equal
 *    sum min(p, q));
 *  - entropy in nats; the top-k probabilities in descending order, ties
 *    broken by the lower token index;
 *  - restricted sampling: per sequence a temperature T_b, a top-k k_b and a
 *    top-p p_b; a row keeps its k_b tokens of largest logit (ties: lower
 *    index first), then, on their renormalised softmax(l / T_b), the
 *    shortest prefix in that order whose probability reaches p_b; the kept
 *    probabilities are renormalised and every other token has probability
 *    0. The accept ratio p'(x)/q'(x) is +inf when q'(x) = 0 < p'(x) and 0
 *    when both are 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_INPUT (-4)

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 [SAL]: ten rounds; each round multiplies counter words 0 and
 * 2 by the two Philox multipliers, xors the high halves into words 1 and 3
 * together with the round key, and permutes; the key is bumped by the two
 * Weyl constants between rounds. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(prod1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)prod1;
        uint32_t n2 = (uint32_t)(prod0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)prod0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

double oracle_u24(uint32_t x) { return (double)(2u * (x >> 9) + 1u) * 0x1p-24; }

double oracle_u52(uint32_t x0, uint32_t x1)
{
    uint64_t k = ((uint64_t)x0 << 20) | (uint64_t)(x1 >> 12);
    return (double)(2u * k + 1u) * 0x1p-53;
}

static void seeded_block(uint64_t seed, uint32_t b, uint32_t i, uint32_t purpose, uint32_t out[4])
{
    uint32_t ctr[4] = {b, i, purpose, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    oracle_philox4x32_10(ctr, key, out);
}

/* accept-test uniform r_i of sequence b, 1-based position i */
double oracle_accept_uniform(uint64_t seed, uint32_t b, uint32_t i)
{
    uint32_t w[4];
    seeded_block(seed, b, i, 0u, w);
    return oracle_u24(w[0]);
}

/* final-draw uniform of sequence b, drawn at 1-based position i = n+1 */
double oracle_draw_uniform(uint64_t seed, uint32_t b, uint32_t i)
{
    uint32_t w[4];
    seeded_block(seed, b, i, 1u, w);
    return oracle_u52(w[0], w[1]);
}

/* ------------------------------------------------------------------------ */
/* element access: dtype 0 = fp32, 1 = bf16 (the top half of an fp32) */
static size_t elem_size(int32_t dtype) { return dtype == 0 ? 4u : 2u; }

static double logit_at(const void *row, int32_t dtype, int64_t v)
{
    if (dtype == 0) return (double)((const float *)row)[v];
    uint32_t bits = (uint32_t)((const uint16_t *)row)[v] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static const void *row_ptr(const void *base, int64_t row, int64_t stride, int32_t dtype)
{
    return (const char *)base + (size_t)row * (size_t)stride * elem_size(dtype);
}

/* Neumaier (improved Kahan-Babuska) compensated sum */
typedef struct { double s, c; } nsum;
static void nsum_add(nsum *a, double x)
{
    double t = a->s + x;
    if (fabs(a->s) >= fabs(x)) a->c += (a->s - t) + x;
    else a->c += (x - t) + a->s;
    a->s = t;
}
static double nsum_get(const nsum *a) { return a->s + a->c; }

/* ------------------------------------------------------------------------ */
/* Temperature softmax normaliser [KAD Part 2; DS App. B.3]:
 * z_v = l_v / T, lse = max z + log sum_v exp(z_v - max z). */
int oracle_row_lse(const void *row, int32_t dtype, int64_t V, double T, double *lse_out)
{
    if (!row || V <= 0 || !(T > 0.0) || !isfinite(T)) return ORACLE_ERR_ARG;
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double l = logit_at(row, dtype, v);
        if (isnan(l) || l == INFINITY) return ORACLE_ERR_INPUT;
        double z = l / T;
        if (z > m) m = z;
    }
    if (m == -INFINITY) return ORACLE_ERR_INPUT;
    nsum s = {0.0, 0.0};
    for (int64_t v = 0; v < V; ++v) nsum_add(&s, exp(logit_at(row, dtype, v) / T - m));
    *lse_out = m + log(nsum_get(&s));
    return ORACLE_OK;
}

/* argmax of the raw logits, lowest index on ties; NaN is a bad input */
int oracle_row_argmax(const void *row, int32_t dtype, int64_t V, int64_t *argmax_out)
{
    if (!row || V <= 0) return ORACLE_ERR_ARG;
    int64_t best = 0;
    double bv = logit_at(row, dtype, 0);
    if (isnan(bv)) return ORACLE_ERR_INPUT;
    for (int64_t v = 1; v < V; ++v) {
        double l = logit_at(row, dtype, v);
        if (isnan(l)) return ORACLE_ERR_INPUT;
        if (l > bv) { bv = l; best = v; }
    }
    *argmax_out = best;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Lenience [DSL]: log f(p, eps) from log p. f_lin(p, eps) = p / eps,
 * f_sq(p, eps) = p / eps^2, f_exp(p, eps) = p^eps; kind 0: f(p) = p. */
#define ORACLE_LENIENCE_NONE 0
#define ORACLE_LENIENCE_LIN 1
#define ORACLE_LENIENCE_SQ 2
#define ORACLE_LENIENCE_EXP 3

static double lenient_log(double log_p, int32_t kind, double eps)
{
    switch (kind) {
    case ORACLE_LENIENCE_LIN: return log_p - log(eps);
    case ORACLE_LENIENCE_SQ: return log_p - 2.0 * log(eps);
    case ORACLE_LENIENCE_EXP: return eps * log_p;
    default: return log_p;
    }
}

static int lenience_ok(int32_t kind, double eps)
{
    if (kind == ORACLE_LENIENCE_NONE) return 1;
    return kind >= ORACLE_LENIENCE_LIN && kind <= ORACLE_LENIENCE_EXP && eps > 0.0 && eps <= 1.0;
}

/* Accept scan [DS Alg. A.1 (rejection thresholds, uniforms, n); LKM rule]:
 * ratio_i = f(p_i(x_i), eps) / q_i(x_i) with p_i = softmax(target_i / T) and
 * q_i = softmax(draft_i / T) (f(p) = p when lossless);
 * n = first i-1 with r_i > ratio_i, else gamma. */
static int32_t accept_scan(const void *p_rows, const void *q_rows, int64_t stride, int32_t dtype,
                           int32_t gamma, const int32_t *x, double T,
                           const double *lse_p, const double *lse_q, const double *r,
                           int32_t len_kind, double eps, double *acc_margin)
{
    for (int32_t i = 0; i < gamma; ++i) {
        const void *pr = row_ptr(p_rows, i, stride, dtype);
        const void *qr = row_ptr(q_rows, i, stride, dtype);
        double log_p = logit_at(pr, dtype, x[i]) / T - lse_p[i];
        double log_q = logit_at(qr, dtype, x[i]) / T - lse_q[i];
        double ratio = exp(lenient_log(log_p, len_kind, eps) - log_q);
        if (acc_margin) acc_margin[i] = fabs(r[i] - ratio);
        if (r[i] > ratio) return i;
    }
    return gamma;
}

/* Final token [DS Alg. A.1, "sample from the adjusted distribution" or
 * "sample from M_p"; KAD steps 4-5]: if n < gamma draw from
 * norm(max(0, p_{n+1} - q_{n+1})), else the bonus token from p_{gamma+1}.
 * Inverse CDF in index order with t = u * R. Returns the token, writes the
 * normalised distance of t to the nearest boundary of the chosen token. */
static int64_t final_draw(const void *p_row, const void *q_row /* NULL: bonus */, int32_t dtype,
                          int64_t V, double T, double lse_p, double lse_q, double u,
                          double *margin_out, int32_t *fallback_out)
{
    double *w = (double *)malloc((size_t)V * sizeof(double));
    if (!w) return -1;
    nsum R = {0.0, 0.0};
    for (int64_t v = 0; v < V; ++v) {
        double log_p = logit_at(p_row, dtype, v) / T - lse_p;
        double p = exp(log_p);
        double wv = p;
        if (q_row) {
            double log_q = logit_at(q_row, dtype, v) / T - lse_q;
            wv = (p == 0.0) ? 0.0 : p * fmax(0.0, -expm1(log_q - log_p));
        }
        w[v] = wv;
        nsum_add(&R, wv);
    }
    int32_t fallback = 0;
    double total = nsum_get(&R);
    if (!(total > 0.0) || !isfinite(total)) {
        /* zero residual mass can only come from rounding: draw from p */
        fallback = 1;
        nsum P = {0.0, 0.0};
        for (int64_t v = 0; v < V; ++v) {
            w[v] = exp(logit_at(p_row, dtype, v) / T - lse_p);
            nsum_add(&P, w[v]);
        }
        total = nsum_get(&P);
    }
    double t = u * total;
    nsum C = {0.0, 0.0};
    double c_prev = 0.0, c_k = 0.0;
    int64_t k = -1;
    for (int64_t v = 0; v < V; ++v) {
        c_prev = nsum_get(&C);
        nsum_add(&C, w[v]);
        c_k = nsum_get(&C);
        if (c_k > t) { k = v; break; }
    }
    if (k < 0) {
        /* t at or past the last boundary through rounding: the last token of
         * positive weight; zero-weight tokens are never chosen */
        for (int64_t v = V - 1; v >= 0; --v)
            if (w[v] > 0.0) { k = v; break; }
        c_prev = c_k = t;
    }
    if (margin_out) {
        double g = fmin(t - c_prev, c_k - t) / total;
        *margin_out = g < 0.0 ? 0.0 : g;
    }
    if (fallback_out) *fallback_out = fallback;
    free(w);
    return k;
}

/* ------------------------------------------------------------------------ */
/* One verify step of one sequence. The draw uniform is `u_fixed`, or, when
 * `seed` is not NULL, the Philox uniform of (seed; sid, n+1, purpose 1),
 * which depends on the n found by the accept scan. */
static int verify_seq_impl(const void *p_rows, const void *q_rows, int64_t row_stride, int32_t dtype,
                           int64_t V, int32_t gamma, const int32_t *x, double T,
                           int32_t len_kind, double eps,
                           const double *r, double u_fixed, const uint64_t *seed, uint32_t sid,
                           int32_t *n_out, int32_t *tokens_out,
                           double *lse_p_out, double *lse_q_out,
                           double *acc_margin_out, double *draw_margin_out, int32_t *fallback_out)
{
    if (!p_rows || (gamma > 0 && (!q_rows || !x || !r)) || gamma < 0 || V <= 0 ||
        row_stride < V || (dtype != 0 && dtype != 1) || !n_out || !tokens_out || !(T > 0.0) ||
        !isfinite(T) || !lenience_ok(len_kind, eps))
        return ORACLE_ERR_ARG;
    for (int32_t i = 0; i <= gamma; ++i) tokens_out[i] = -1;
    *n_out = -1;
    for (int32_t i = 0; i < gamma; ++i)
        if (x[i] < 0 || (int64_t)x[i] >= V) return ORACLE_ERR_INPUT;

    double *lse_p = (double *)malloc(sizeof(double) * (size_t)(2 * gamma + 1));
    if (!lse_p) return ORACLE_ERR_ARG;
    double *lse_q = lse_p + gamma + 1;
    int rc = ORACLE_OK;
    for (int32_t i = 0; i <= gamma && rc == ORACLE_OK; ++i)
        rc = oracle_row_lse(row_ptr(p_rows, i, row_stride, dtype), dtype, V, T, &lse_p[i]);
    for (int32_t i = 0; i < gamma && rc == ORACLE_OK; ++i)
        rc = oracle_row_lse(row_ptr(q_rows, i, row_stride, dtype), dtype, V, T, &lse_q[i]);
    if (rc != ORACLE_OK) { free(lse_p); return rc; }
    if (lse_p_out) memcpy(lse_p_out, lse_p, sizeof(double) * (size_t)(gamma + 1));
    if (lse_q_out && gamma > 0) memcpy(lse_q_out, lse_q, sizeof(double) * (size_t)gamma);

    int32_t n = accept_scan(p_rows, q_rows, row_stride, dtype, gamma, x, T, lse_p, lse_q, r,
                            len_kind, eps, acc_margin_out);
    double u = seed ? oracle_draw_uniform(*seed, sid, (uint32_t)(n + 1)) : u_fixed;
    const void *p_row = row_ptr(p_rows, n, row_stride, dtype);
    const void *q_row = (n < gamma) ? row_ptr(q_rows, n, row_stride, dtype) : NULL;
    int64_t k = final_draw(p_row, q_row, dtype, V, T, lse_p[n], n < gamma ? lse_q[n] : 0.0, u,
                           draw_margin_out, fallback_out);
    free(lse_p);
    if (k < 0) return ORACLE_ERR_ARG;
    for (int32_t i = 0; i < n; ++i) tokens_out[i] = x[i];
    tokens_out[n] = (int32_t)k;
    *n_out = n;
    return ORACLE_OK;
}

/* One sequence with explicit uniforms r[0..gamma-1] (accept tests) and u
 * (final draw). p_rows holds gamma+1 target rows, q_rows gamma draft rows,
 * both `row_stride` elements apart. tokens_out gets gamma+1 slots:
 * x_1..x_n, the final token, then -1. Optional outputs may be NULL. */
int oracle_verify_seq_u(const void *p_rows, const void *q_rows, int64_t row_stride, int32_t dtype,
                        int64_t V, int32_t gamma, const int32_t *x, double T,
                        const double *r, double u,
                        int32_t *n_out, int32_t *tokens_out,
                        double *lse_p_out, double *lse_q_out,
                        double *acc_margin_out, double *draw_margin_out, int32_t *fallback_out)
{
    return verify_seq_impl(p_rows, q_rows, row_stride, dtype, V, gamma, x, T,
                           ORACLE_LENIENCE_NONE, 1.0, r, u, NULL, 0u,
                           n_out, tokens_out, lse_p_out, lse_q_out, acc_margin_out,
                           draw_margin_out, fallback_out);
}

/* The same with lenience [DSL]: len_kind 0..3, eps in (0, 1]. */
int oracle_verify_seq_u_lenient(const void *p_rows, const void *q_rows, int64_t row_stride,
                                int32_t dtype, int64_t V, int32_t gamma, const int32_t *x,
                                double T, int32_t len_kind, double eps,
                                const double *r, double u, int32_t *n_out, int32_t *tokens_out,
                                double *acc_margin_out, double *draw_margin_out)
{
    return verify_seq_impl(p_rows, q_rows, row_stride, dtype, V, gamma, x, T, len_kind, eps, r,
                           u, NULL, 0u, n_out, tokens_out, NULL, NULL, acc_margin_out,
                           draw_margin_out, NULL);
}

/* Greedy verify of one sequence [KAD "Greedy vs sampling"]: a_i = argmax p_i;
 * n = first i-1 with x_i != a_i, else gamma; tokens x_1..x_n, a_{n+1}. */
int oracle_verify_greedy_seq(const void *p_rows, int64_t row_stride, int32_t dtype, int64_t V,
                             int32_t gamma, const int32_t *x, int32_t *n_out, int32_t *tokens_out)
{
    if (!p_rows || gamma < 0 || (gamma > 0 && !x) || V <= 0 || row_stride < V ||
        (dtype != 0 && dtype != 1) || !n_out || !tokens_out)
        return ORACLE_ERR_ARG;
    for (int32_t i = 0; i <= gamma; ++i) tokens_out[i] = -1;
    *n_out = -1;
    for (int32_t i = 0; i < gamma; ++i)
        if (x[i] < 0 || (int64_t)x[i] >= V) return ORACLE_ERR_INPUT;
    int32_t n = gamma;
    int64_t a = 0;
    for (int32_t i = 0; i <= gamma; ++i) {
        int rc = oracle_row_argmax(row_ptr(p_rows, i, row_stride, dtype), dtype, V, &a);
        if (rc != ORACLE_OK) return rc;
        if (i == gamma || (int64_t)x[i] != a) { n = i; break; }
    }
    for (int32_t i = 0; i < n; ++i) tokens_out[i] = x[i];
    tokens_out[n] = (int32_t)a;
    *n_out = n;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Batch over sequences in the library's ragged layout (host pointers):
 *   p_{b,i} (i = 1..gamma_b+1) is row p_row_off[b] + i-1 of `target`,
 *   q_{b,i} (i = 1..gamma_b)   is row q_row_off[b] + i-1 of `draft`,
 *   x_{b,i} is draft_tokens[b*gamma_max + i-1].
 * The Philox counter uses seq_ids[b] (or b when seq_ids is NULL), so a subset
 * of a larger batch reproduces that batch's draws. Sequences with invalid
 * input get n = -1 and all tokens -1; the call then returns ORACLE_ERR_INPUT.
 * T <= 0 selects the greedy verify. */
typedef struct {
    const void *target, *draft;
    int64_t stride, V, target_rows, draft_rows;
    int32_t dtype, B, gamma_max;
    const int64_t *p_off, *q_off;
    const int32_t *tokens, *gamma, *seq_ids;
    double T;
    int32_t len_kind;
    double eps;
    uint64_t seed;
    int32_t *n_out, *tok_out;
    double *lse_p, *lse_q, *acc_margin, *draw_margin;
    int32_t *fallback;
    int32_t nthreads, tid;
    int rc;
} batch_job;

static void verify_one_of_batch(batch_job *J, int32_t b)
{
    int32_t gm = J->gamma_max;
    int32_t *tok = J->tok_out + (size_t)b * (size_t)(gm + 1);
    for (int32_t i = 0; i <= gm; ++i) tok[i] = -1;
    J->n_out[b] = -1;
    int32_t g = J->gamma[b];
    int sampling = J->T > 0.0;
    if (g < 0 || g > gm || J->p_off[b] < 0 || J->p_off[b] + g + 1 > J->target_rows ||
        (sampling && g > 0 && (J->q_off[b] < 0 || J->q_off[b] + g > J->draft_rows))) {
        J->rc = ORACLE_ERR_INPUT;
        return;
    }
    const void *p_rows = row_ptr(J->target, J->p_off[b], J->stride, J->dtype);
    const int32_t *x = J->tokens + (size_t)b * (size_t)gm;
    int32_t n = -1;
    int rc;
    if (!sampling) {
        rc = oracle_verify_greedy_seq(p_rows, J->stride, J->dtype, J->V, g, x, &n, tok);
    } else {
        const void *q_rows = g > 0 ? row_ptr(J->draft, J->q_off[b], J->stride, J->dtype) : p_rows;
        uint32_t sid = J->seq_ids ? (uint32_t)J->seq_ids[b] : (uint32_t)b;
        double r[512], lp[513], lq[512], am[512];
        if (g > 512) { J->rc = ORACLE_ERR_ARG; return; }
        for (int32_t i = 0; i < g; ++i) {
            r[i] = oracle_accept_uniform(J->seed, sid, (uint32_t)(i + 1));
            am[i] = NAN;
        }
        double dm = NAN;
        int32_t fb = 0;
        rc = verify_seq_impl(p_rows, q_rows, J->stride, J->dtype, J->V, g, x, J->T, J->len_kind,
                             J->eps, r, 0.0, &J->seed, sid, &n, tok, lp, lq, am, &dm, &fb);
        if (rc == ORACLE_OK) {
            if (J->lse_p) {
                double *o = J->lse_p + (size_t)b * (size_t)(gm + 1);
                for (int32_t i = 0; i <= gm; ++i) o[i] = i <= g ? lp[i] : NAN;
            }
            if (J->lse_q && gm > 0) {
                double *o = J->lse_q + (size_t)b * (size_t)gm;
                for (int32_t i = 0; i < gm; ++i) o[i] = i < g ? lq[i] : NAN;
            }
            if (J->acc_margin && gm > 0) {
                double *o = J->acc_margin + (size_t)b * (size_t)gm;
                for (int32_t i = 0; i < gm; ++i) o[i] = i < g ? am[i] : NAN;
            }
            if (J->draw_margin) J->draw_margin[b] = dm;
            if (J->fallback) J->fallback[b] = fb;
        }
    }
    if (rc != ORACLE_OK) {
        for (int32_t i = 0; i <= gm; ++i) tok[i] = -1;
        J->n_out[b] = -1;
        J->rc = rc == ORACLE_ERR_ARG ? ORACLE_ERR_ARG : ORACLE_ERR_INPUT;
        return;
    }
    J->n_out[b] = n;
}

static void *batch_worker(void *arg)
{
    batch_job *J = (batch_job *)arg;
    for (int32_t b = J->tid; b < J->B; b += J->nthreads) verify_one_of_batch(J, b);
    return NULL;
}

int oracle_verify_batch_lenient(const void *target, const void *draft, int64_t row_stride,
                                int32_t dtype, int64_t V, int64_t target_rows, int64_t draft_rows,
                                int32_t B, int32_t gamma_max,
                                const int64_t *p_row_off, const int64_t *q_row_off,
                                const int32_t *draft_tokens, const int32_t *gamma,
                                const int32_t *seq_ids, double T, int32_t len_kind, double eps,
                                uint64_t seed,
                        int32_t *n_out, int32_t *tokens_out,
                        double *lse_p_out, double *lse_q_out,
                        double *acc_margin_out, double *draw_margin_out, int32_t *fallback_out,
                        int32_t nthreads)
{
    int sampling = T > 0.0;
    if (B < 0 || gamma_max < 0 || gamma_max > 512 || V <= 0 || row_stride < V ||
        (dtype != 0 && dtype != 1) || !target || !p_row_off || !gamma || !n_out || !tokens_out ||
        (gamma_max > 0 && !draft_tokens) || (sampling && gamma_max > 0 && (!draft || !q_row_off)) ||
        !isfinite(T) || (sampling && !lenience_ok(len_kind, eps)))
        return ORACLE_ERR_ARG;
    if (B == 0) return ORACLE_OK;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B) nthreads = B;
    if (nthreads > 256) nthreads = 256;
    batch_job jobs[256];
    pthread_t th[256];
    for (int32_t t = 0; t < nthreads; ++t) {
        batch_job J = {target, draft, row_stride, V, target_rows, draft_rows, dtype, B, gamma_max,
                       p_row_off, q_row_off, draft_tokens, gamma, seq_ids, T, len_kind, eps,
                       seed, n_out,
                       tokens_out, lse_p_out, lse_q_out, acc_margin_out, draw_margin_out,
                       fallback_out, nthreads, t, ORACLE_OK};
        jobs[t] = J;
    }
    int started = 0;
    for (int32_t t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, batch_worker, &jobs[t]) == 0) started = t;
        else break;
    /* any thread that failed to start has its share done here */
    batch_worker(&jobs[0]);
    for (int32_t t = started + 1; t < nthreads; ++t) batch_worker(&jobs[t]);
    for (int32_t t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    int rc = ORACLE_OK;
    for (int32_t t = 0; t < nthreads; ++t)
        if (jobs[t].rc == ORACLE_ERR_ARG) rc = ORACLE_ERR_ARG;
        else if (jobs[t].rc != ORACLE_OK && rc == ORACLE_OK) rc = jobs[t].rc;
    return rc;
}

/* The lossless batch call (lenience kind 0). */
int oracle_verify_batch(const void *target, const void *draft, int64_t row_stride, int32_t dtype,
                        int64_t V, int64_t target_rows, int64_t draft_rows,
                        int32_t B, int32_t gamma_max,
                        const int64_t *p_row_off, const int64_t *q_row_off,
                        const int32_t *draft_tokens, const int32_t *gamma, const int32_t *seq_ids,
                        double T, uint64_t seed,
                        int32_t *n_out, int32_t *tokens_out,
                        double *lse_p_out, double *lse_q_out,
                        double *acc_margin_out, double *draw_margin_out, int32_t *fallback_out,
                        int32_t nthreads)
{
    return oracle_verify_batch_lenient(target, draft, row_stride, dtype, V, target_rows,
                                       draft_rows, B, gamma_max, p_row_off, q_row_off,
                                       draft_tokens, gamma, seq_ids, T, ORACLE_LENIENCE_NONE, 1.0,
                                       seed, n_out, tokens_out, lse_p_out, lse_q_out,
                                       acc_margin_out, draw_margin_out, fallback_out, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Acceptance statistics of one position [DSB]: with p = softmax(target / T)
 * and q = softmax(draft / T), beta = sum_v min(p_v, q_v) -- the probability
 * that the accept test passes when the draft token is drawn from q -- and
 * TVD = 1/2 sum_v |p_v - q_v|. */
int oracle_pair_stats(const void *p_row, const void *q_row, int32_t dtype, int64_t V, double T,
                      double *beta_out, double *tvd_out)
{
    if (!p_row || !q_row || V <= 0 || !beta_out || !tvd_out) return ORACLE_ERR_ARG;
    double lse_p, lse_q;
    int rc = oracle_row_lse(p_row, dtype, V, T, &lse_p);
    if (rc == ORACLE_OK) rc = oracle_row_lse(q_row, dtype, V, T, &lse_q);
    if (rc != ORACLE_OK) return rc;
    nsum b = {0.0, 0.0}, d = {0.0, 0.0};
    for (int64_t v = 0; v < V; ++v) {
        double p = exp(logit_at(p_row, dtype, v) / T - lse_p);
        double q = exp(logit_at(q_row, dtype, v) / T - lse_q);
        nsum_add(&b, fmin(p, q));
        nsum_add(&d, fabs(p - q));
    }
    *beta_out = nsum_get(&b);
    *tvd_out = 0.5 * nsum_get(&d);
    return ORACLE_OK;
}

/* Draft-distribution features of one row [DIS Eq. 2, App. D.1]:
 * q = softmax(row / T); entropy = -sum_v q_v log q_v in nats (a token of
 * probability 0 adds nothing); the k largest q_v in descending order with
 * their token indices, ties to the lower index (compared on the raw logits,
 * which order the same way as q); slots past V get probability 0, index -1. */
int oracle_row_features(const void *row, int32_t dtype, int64_t V, double T, int32_t k,
                        double *entropy_out, double *topk_prob, int64_t *topk_idx)
{
    if (!row || V <= 0 || k < 0 || !entropy_out || (k > 0 && (!topk_prob || !topk_idx)))
        return ORACLE_ERR_ARG;
    double lse;
    int rc = oracle_row_lse(row, dtype, V, T, &lse);
    if (rc != ORACLE_OK) return rc;
    nsum h = {0.0, 0.0};
    for (int64_t v = 0; v < V; ++v) {
        double l = logit_at(row, dtype, v);
        if (l == -INFINITY) continue;
        double log_q = l / T - lse;
        nsum_add(&h, -exp(log_q) * log_q);
    }
    *entropy_out = nsum_get(&h);
    /* selection by insertion into a list kept sorted (value desc, index asc) */
    int32_t kept = 0;
    for (int64_t v = 0; v < V && k > 0; ++v) {
        double l = logit_at(row, dtype, v);
        if (kept == k && !(l > logit_at(row, dtype, topk_idx[k - 1]))) continue;
        int32_t at = kept < k ? kept : k - 1;
        while (at > 0 && l > logit_at(row, dtype, topk_idx[at - 1])) {
            topk_idx[at] = topk_idx[at - 1];
            --at;
        }
        topk_idx[at] = v;
        if (kept < k) ++kept;
    }
    for (int32_t j = 0; j < k; ++j) {
        if (j < kept) {
            topk_prob[j] = exp(logit_at(row, dtype, topk_idx[j]) / T - lse);
        } else {
            topk_prob[j] = 0.0;
            topk_idx[j] = -1;
        }
    }
    return ORACLE_OK;
}

/* Both per-row functions above over a batch, threaded over sequences (or
 * rows): beta and TVD of the positions i = 1..gamma_b of every sequence, in
 * the batch layout of oracle_verify_batch ([B, gamma_max], NaN past gamma_b
 * or for a sequence with bad input); entropy and top-k of `nrows` rows. */
typedef struct {
    const void *target, *draft;
    int64_t stride, V, target_rows, draft_rows;
    int32_t dtype, B, gamma_max, k;
    const int64_t *p_off, *q_off;
    const int32_t *gamma;
    double T;
    double *beta, *tvd, *entropy, *topk_prob;
    int64_t *topk_idx;
    int32_t nthreads, tid;
    int rc;
} stats_job;

static void *pair_stats_worker(void *arg)
{
    stats_job *J = (stats_job *)arg;
    for (int32_t b = J->tid; b < J->B; b += J->nthreads) {
        int32_t gm = J->gamma_max, g = J->gamma[b];
        for (int32_t i = 0; i < gm; ++i) {
            J->beta[(size_t)b * gm + i] = NAN;
            J->tvd[(size_t)b * gm + i] = NAN;
        }
        if (g < 0 || g > gm || J->p_off[b] < 0 || J->p_off[b] + g + 1 > J->target_rows ||
            (g > 0 && (J->q_off[b] < 0 || J->q_off[b] + g > J->draft_rows))) {
            J->rc = ORACLE_ERR_INPUT;
            continue;
        }
        double be[512], tv[512];
        for (int32_t i = 0; i < g; ++i) {
            int rc = oracle_pair_stats(row_ptr(J->target, J->p_off[b] + i, J->stride, J->dtype),
                                       row_ptr(J->draft, J->q_off[b] + i, J->stride, J->dtype),
                                       J->dtype, J->V, J->T, &be[i], &tv[i]);
            if (rc != ORACLE_OK) {
                J->rc = rc;
                g = -1;
                break;
            }
        }
        for (int32_t i = 0; i < g; ++i) {
            J->beta[(size_t)b * gm + i] = be[i];
            J->tvd[(size_t)b * gm + i] = tv[i];
        }
    }
    return NULL;
}

static void *features_worker(void *arg)
{
    stats_job *J = (stats_job *)arg;
    for (int32_t r = J->tid; r < J->B; r += J->nthreads) {
        int rc = oracle_row_features(row_ptr(J->target, r, J->stride, J->dtype), J->dtype, J->V,
                                     J->T, J->k, &J->entropy[r],
                                     J->topk_prob + (size_t)r * J->k,
                                     J->topk_idx + (size_t)r * J->k);
        if (rc != ORACLE_OK) {
            J->entropy[r] = NAN;
            for (int32_t j = 0; j < J->k; ++j) {
                J->topk_prob[(size_t)r * J->k + j] = NAN;
                J->topk_idx[(size_t)r * J->k + j] = -1;
            }
            J->rc = rc;
        }
    }
    return NULL;
}

static int run_stats_jobs(stats_job *proto, int32_t units, void *(*worker)(void *))
{
    int32_t nthreads = proto->nthreads;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > units) nthreads = units;
    if (nthreads > 256) nthreads = 256;
    if (nthreads < 1) return ORACLE_OK;
    stats_job jobs[256];
    pthread_t th[256];
    for (int32_t t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].nthreads = nthreads;
        jobs[t].tid = t;
        jobs[t].rc = ORACLE_OK;
    }
    int started = 0;
    for (int32_t t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, worker, &jobs[t]) == 0) started = t;
        else break;
    worker(&jobs[0]);
    for (int32_t t = started + 1; t < nthreads; ++t) worker(&jobs[t]);
    for (int32_t t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    int rc = ORACLE_OK;
    for (int32_t t = 0; t < nthreads; ++t)
        if (jobs[t].rc != ORACLE_OK && rc == ORACLE_OK) rc = jobs[t].rc;
    return rc;
}

int oracle_pair_stats_batch(const void *target, const void *draft, int64_t row_stride,
                            int32_t dtype, int64_t V, int64_t target_rows, int64_t draft_rows,
                            int32_t B, int32_t gamma_max, const int64_t *p_row_off,
                            const int64_t *q_row_off, const int32_t *gamma, double T,
                            double *beta_out, double *tvd_out, int32_t nthreads)
{
    if (B < 0 || gamma_max < 0 || gamma_max > 512 || V <= 0 || row_stride < V ||
        (dtype != 0 && dtype != 1) || !(T > 0.0) || !isfinite(T) ||
        (B > 0 && (!target || !draft || !p_row_off || !q_row_off || !gamma ||
                   (gamma_max > 0 && (!beta_out || !tvd_out)))))
        return ORACLE_ERR_ARG;
    stats_job J = {target, draft, row_stride, V, target_rows, draft_rows, dtype, B, gamma_max, 0,
                   p_row_off, q_row_off, gamma, T, beta_out, tvd_out, NULL, NULL, NULL,
                   nthreads, 0, ORACLE_OK};
    return run_stats_jobs(&J, B, pair_stats_worker);
}

int oracle_row_features_batch(const void *rows, int64_t row_stride, int32_t dtype, int64_t V,
                              int32_t nrows, double T, int32_t k, double *entropy_out,
                              double *topk_prob, int64_t *topk_idx, int32_t nthreads)
{
    if (nrows < 0 || V <= 0 || row_stride < V || (dtype != 0 && dtype != 1) || k < 0 ||
        !(T > 0.0) || !isfinite(T) ||
        (nrows > 0 && (!rows || !entropy_out || (k > 0 && (!topk_prob || !topk_idx)))))
        return ORACLE_ERR_ARG;
    stats_job J = {rows, NULL, row_stride, V, nrows, 0, dtype, nrows, 0, k, NULL, NULL, NULL, T,
                   NULL, NULL, entropy_out, topk_prob, topk_idx, nthreads, 0, ORACLE_OK};
    return run_stats_jobs(&J, nrows, features_worker);
}

/* ------------------------------------------------------------------------ */
/* Restricted sampling [KGS]: the restricted distribution of one row, as
 * probabilities prob[0..V) (0 outside the kept set). Returns the number of
 * kept tokens, or a negative error code. */
static int64_t restricted_row(const void *row, int32_t dtype, int64_t V, double T, int32_t k,
                              double top_p, double *prob, int64_t *idx /* scratch [k] */,
                              double *w /* scratch [k] */)
{
    if (k > V) k = (int32_t)V;
    int32_t kept = 0;
    for (int64_t v = 0; v < V; ++v) {
        double l = logit_at(row, dtype, v);
        if (isnan(l) || l == INFINITY) return ORACLE_ERR_INPUT;
        if (kept == k && !(l > logit_at(row, dtype, idx[k - 1]))) continue;
        int32_t at = kept < k ? kept : k - 1;
        while (at > 0 && l > logit_at(row, dtype, idx[at - 1])) {
            idx[at] = idx[at - 1];
            --at;
        }
        idx[at] = v;
        if (kept < k) ++kept;
    }
    double l0 = logit_at(row, dtype, idx[0]);
    if (l0 == -INFINITY) return ORACLE_ERR_INPUT;
    double total = 0.0;
    for (int32_t j = 0; j < kept; ++j) {
        w[j] = exp(logit_at(row, dtype, idx[j]) / T - l0 / T);
        total += w[j];
    }
    /* the shortest prefix whose renormalised probability reaches top_p */
    int32_t m = 0;
    double run = 0.0;
    while (m < kept) {
        run += w[m];
        ++m;
        if (run / total >= top_p) break;
    }
    double z = 0.0;
    for (int32_t j = 0; j < m; ++j) z += w[j];
    for (int64_t v = 0; v < V; ++v) prob[v] = 0.0;
    for (int32_t j = 0; j < m; ++j) prob[idx[j]] = w[j] / z;
    return m;
}

/* Inverse-CDF draw from weights w[0..V) in index order at t = u * R
 * (R = sum w); zero-weight tokens are never drawn. Returns the token and the
 * normalised distance of t to the nearest boundary of its interval. */
static int64_t draw_from_weights(const double *w, int64_t V, double u, double *margin_out)
{
    nsum R = {0.0, 0.0};
    for (int64_t v = 0; v < V; ++v) nsum_add(&R, w[v]);
    double total = nsum_get(&R);
    double t = u * total;
    nsum C = {0.0, 0.0};
    double c_prev = 0.0, c_k = 0.0;
    int64_t k = -1;
    for (int64_t v = 0; v < V; ++v) {
        c_prev = nsum_get(&C);
        nsum_add(&C, w[v]);
        c_k = nsum_get(&C);
        if (c_k > t) { k = v; break; }
    }
    if (k < 0) {
        for (int64_t v = V - 1; v >= 0; --v)
            if (w[v] > 0.0) { k = v; break; }
        c_prev = c_k = t;
    }
    if (margin_out) {
        double g = fmin(t - c_prev, c_k - t) / total;
        *margin_out = g < 0.0 ? 0.0 : g;
    }
    return k;
}

/* One sequence of a restricted verify: p_{i} and q_{i} replaced by their
 * restricted distributions; the accept scan ([DS Alg. A.1; LKM rule]) with
 * the ratio p'(x)/q'(x), then the residual norm(max(0, p' - q')) after a
 * rejection or the bonus token from p'_{gamma+1}. The accept uniforms are
 * r[0..gamma) when given, else the seeded ones; the draw uniform is u_fixed
 * when seed is NULL, else the seeded one at n + 1. */
static int verify_seq_restricted(const void *p_rows, const void *q_rows, int64_t stride,
                                 int32_t dtype, int64_t V, int32_t gamma, const int32_t *x,
                                 double T, int32_t topk, double topp, const double *r,
                                 double u_fixed, const uint64_t *seed, uint32_t sid,
                                 int32_t *n_out, int32_t *tokens_out, double *acc_margin,
                                 double *draw_margin)
{
    for (int32_t i = 0; i <= gamma; ++i) tokens_out[i] = -1;
    *n_out = -1;
    if (!(T > 0.0) || !isfinite(T) || topk < 1 || !(topp > 0.0) || !(topp <= 1.0))
        return ORACLE_ERR_INPUT;
    for (int32_t i = 0; i < gamma; ++i)
        if (x[i] < 0 || (int64_t)x[i] >= V) return ORACLE_ERR_INPUT;
    int32_t k = topk > V ? (int32_t)V : topk;
    double *pp = (double *)malloc(sizeof(double) * (size_t)V * 3 + sizeof(double) * (size_t)k);
    int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)k);
    if (!pp || !idx) { free(pp); free(idx); return ORACLE_ERR_ARG; }
    double *qq = pp + V, *w = qq + V, *ws = w + V;
    int rc = ORACLE_OK;
    /* every row of the sequence is validated, as the lossless path does */
    for (int32_t i = 0; i <= gamma && rc == ORACLE_OK; ++i)
        if (restricted_row(row_ptr(p_rows, i, stride, dtype), dtype, V, T, k, topp, w, idx, ws) < 0)
            rc = ORACLE_ERR_INPUT;
    for (int32_t i = 0; i < gamma && rc == ORACLE_OK; ++i)
        if (restricted_row(row_ptr(q_rows, i, stride, dtype), dtype, V, T, k, topp, w, idx, ws) < 0)
            rc = ORACLE_ERR_INPUT;
    int32_t n = gamma;
    for (int32_t i = 0; i < gamma && rc == ORACLE_OK; ++i) {
        restricted_row(row_ptr(p_rows, i, stride, dtype), dtype, V, T, k, topp, pp, idx, ws);
        restricted_row(row_ptr(q_rows, i, stride, dtype), dtype, V, T, k, topp, qq, idx, ws);
        double pv = pp[x[i]], qv = qq[x[i]];
        double ratio = qv > 0.0 ? pv / qv : (pv > 0.0 ? INFINITY : 0.0);
        double ri = r ? r[i] : oracle_accept_uniform(*seed, sid, (uint32_t)(i + 1));
        if (acc_margin) acc_margin[i] = fabs(ri - ratio);
        if (ri > ratio) {
            n = i;
            break;
        }
    }
    if (rc == ORACLE_OK) {
        restricted_row(row_ptr(p_rows, n, stride, dtype), dtype, V, T, k, topp, pp, idx, ws);
        if (n < gamma) {
            restricted_row(row_ptr(q_rows, n, stride, dtype), dtype, V, T, k, topp, qq, idx, ws);
            double R = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                w[v] = fmax(0.0, pp[v] - qq[v]);
                R += w[v];
            }
            if (!(R > 0.0))  /* zero residual mass through rounding: draw from p' */
                for (int64_t v = 0; v < V; ++v) w[v] = pp[v];
        } else {
            for (int64_t v = 0; v < V; ++v) w[v] = pp[v];
        }
        double u = seed ? oracle_draw_uniform(*seed, sid, (uint32_t)(n + 1)) : u_fixed;
        int64_t tok = draw_from_weights(w, V, u, draw_margin);
        for (int32_t i = 0; i < n; ++i) tokens_out[i] = x[i];
        tokens_out[n] = (int32_t)tok;
        *n_out = n;
    }
    free(pp);
    free(idx);
    return rc;
}

typedef struct {
    const void *target, *draft;
    int64_t stride, V, target_rows, draft_rows;
    int32_t dtype, B, gamma_max;
    const int64_t *p_off, *q_off;
    const int32_t *tokens, *gamma, *seq_ids, *topk;
    const double *T, *topp;
    uint64_t seed;
    int32_t *n_out, *tok_out;
    double *acc_margin, *draw_margin;
    int32_t nthreads, tid;
    int rc;
} restricted_job;

static void *restricted_worker(void *arg)
{
    restricted_job *J = (restricted_job *)arg;
    for (int32_t b = J->tid; b < J->B; b += J->nthreads) {
        int32_t gm = J->gamma_max, g = J->gamma[b];
        int32_t *tok = J->tok_out + (size_t)b * (size_t)(gm + 1);
        for (int32_t i = 0; i <= gm; ++i) tok[i] = -1;
        J->n_out[b] = -1;
        if (J->acc_margin)
            for (int32_t i = 0; i < gm; ++i) J->acc_margin[(size_t)b * gm + i] = NAN;
        if (J->draw_margin) J->draw_margin[b] = NAN;
        if (g < 0 || g > gm || J->p_off[b] < 0 || J->p_off[b] + g + 1 > J->target_rows ||
            (g > 0 && (J->q_off[b] < 0 || J->q_off[b] + g > J->draft_rows))) {
            J->rc = ORACLE_ERR_INPUT;
            continue;
        }
        const void *p_rows = row_ptr(J->target, J->p_off[b], J->stride, J->dtype);
        const void *q_rows = g > 0 ? row_ptr(J->draft, J->q_off[b], J->stride, J->dtype) : p_rows;
        uint32_t sid = J->seq_ids ? (uint32_t)J->seq_ids[b] : (uint32_t)b;
        int32_t n = -1;
        int rc = verify_seq_restricted(p_rows, q_rows, J->stride, J->dtype, J->V, g,
                                       J->tokens + (size_t)b * gm, J->T[b], J->topk[b],
                                       J->topp ? J->topp[b] : 1.0, NULL, 0.0, &J->seed, sid,
                                       &n, tok,
                                       J->acc_margin ? J->acc_margin + (size_t)b * gm : NULL,
                                       J->draw_margin ? J->draw_margin + b : NULL);
        if (rc != ORACLE_OK) {
            for (int32_t i = 0; i <= gm; ++i) tok[i] = -1;
            J->rc = rc;
            continue;
        }
        J->n_out[b] = n;
    }
    return NULL;
}

/* The restricted verify over a batch in the library's ragged layout: per
 * sequence temperature T[b], top-k topk[b] >= 1 and top-p topp[b] in (0, 1]
 * (NULL: 1). A sequence with bad input or parameters gets n = -1. */
int oracle_verify_batch_restricted(const void *target, const void *draft, int64_t row_stride,
                                   int32_t dtype, int64_t V, int64_t target_rows,
                                   int64_t draft_rows, int32_t B, int32_t gamma_max,
                                   const int64_t *p_row_off, const int64_t *q_row_off,
                                   const int32_t *draft_tokens, const int32_t *gamma,
                                   const int32_t *seq_ids, const double *T, const int32_t *topk,
                                   const double *topp, uint64_t seed, int32_t *n_out,
                                   int32_t *tokens_out, double *acc_margin_out,
                                   double *draw_margin_out, int32_t nthreads)
{
    if (B < 0 || gamma_max < 0 || V <= 0 || row_stride < V || (dtype != 0 && dtype != 1) ||
        (B > 0 && (!target || !draft || !p_row_off || !q_row_off || !gamma || !T || !topk ||
                   !n_out || !tokens_out || (gamma_max > 0 && !draft_tokens))))
        return ORACLE_ERR_ARG;
    if (B == 0) return ORACLE_OK;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B) nthreads = B;
    if (nthreads > 256) nthreads = 256;
    restricted_job jobs[256];
    pthread_t th[256];
    for (int32_t t = 0; t < nthreads; ++t) {
        restricted_job J = {target, draft, row_stride, V, target_rows, draft_rows, dtype, B,
                            gamma_max, p_row_off, q_row_off, draft_tokens, gamma, seq_ids, topk,
                            T, topp, seed, n_out, tokens_out, acc_margin_out, draw_margin_out,
                            nthreads, t, ORACLE_OK};
        jobs[t] = J;
    }
    int started = 0;
    for (int32_t t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, restricted_worker, &jobs[t]) == 0) started = t;
        else break;
    restricted_worker(&jobs[0]);
    for (int32_t t = started + 1; t < nthreads; ++t) restricted_worker(&jobs[t]);
    for (int32_t t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    int rc = ORACLE_OK;
    for (int32_t t = 0; t < nthreads; ++t)
        if (jobs[t].rc != ORACLE_OK && rc == ORACLE_OK) rc = jobs[t].rc;
    return rc;
}

/* One sequence of the restricted verify with explicit uniforms (the exact
 * enumeration pins integrate over them): r[0..gamma) accept tests, u draw. */
int oracle_verify_seq_restricted_u(const void *p_rows, const void *q_rows, int64_t row_stride,
                                   int32_t dtype, int64_t V, int32_t gamma, const int32_t *x,
                                   double T, int32_t topk, double topp, const double *r,
                                   double u, int32_t *n_out, int32_t *tokens_out)
{
    if (!p_rows || !q_rows || gamma < 0 || (gamma > 0 && (!x || !r)) || V <= 0 ||
        row_stride < V || !n_out || !tokens_out)
        return ORACLE_ERR_ARG;
    return verify_seq_restricted(p_rows, q_rows, row_stride, dtype, V, gamma, x, T, topk, topp,
                                 r, u, NULL, 0u, n_out, tokens_out, NULL, NULL);
}

/* The restricted distribution of one row, for the pins. */
int oracle_restricted_row(const void *row, int32_t dtype, int64_t V, double T, int32_t topk,
                          double topp, double *prob_out)
{
    if (!row || V <= 0 || topk < 1 || !(T > 0.0) || !(topp > 0.0) || !(topp <= 1.0) || !prob_out)
        return ORACLE_ERR_ARG;
    int32_t k = topk > V ? (int32_t)V : topk;
    int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)k);
    double *ws = (double *)malloc(sizeof(double) * (size_t)k);
    if (!idx || !ws) { free(idx); free(ws); return ORACLE_ERR_ARG; }
    int64_t m = restricted_row(row, dtype, V, T, k, topp, prob_out, idx, ws);
    free(idx);
    free(ws);
    return m < 0 ? (int)m : ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Block efficiency under i.i.d. acceptance [DS Sec. 3 "block efficiency";
 * KAD "Speedup math"]: tau = (1 - alpha^(gamma+1)) / (1 - alpha). */
double oracle_block_efficiency(double alpha, int32_t gamma)
{
    if (alpha == 1.0) return (double)gamma + 1.0;
    return (1.0 - pow(alpha, (double)gamma + 1.0)) / (1.0 - alpha);
}

/* Expected tokens emitted by one verify step when position i is accepted
 * with probability beta[i-1] independently: sum_{k=0..gamma} P(n >= k)
 * = 1 + sum_{k=1..gamma} prod_{i<=k} beta_i. The i.i.d. case is the formula
 * above. */
double oracle_expected_emitted(const double *beta, int32_t gamma)
{
    double e = 1.0, run = 1.0;
    for (int32_t k = 0; k < gamma; ++k) {
        run *= beta[k];
        e += run;
    }
    return e;
}
