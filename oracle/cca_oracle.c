/*
 * CCA prefill oracle: a plain, slow, fp64 CPU evaluation of the two formulas
 * of Core Context Aware attention.  TEST INFRASTRUCTURE ONLY: the test suite,
 * the smoke check and the timed CPU baseline call it; the product path never
 * does.  It shares no code, header or constant with the CUDA library.
 *
 * Sources (page titles as published):
 *  - "Core Context Aware Transformers for Long Context Language Modeling"
 *    (digest.lyk-ai.com, Method section): the global-aware pooling equation
 *        c_i = softmax(Q_{ig} K'_{I_i}^T / sqrt(d)) X^G_{I_i}
 *    and the fusion equation
 *        Att_i = softmax(Q_i [K^G_{T_i}; K^L_{U_i}]^T / sqrt(d)) [V^G_{T_i}; V^L_{U_i}].
 *  - The same paper's news write-up (changsha.jmyizhao.com): groups are
 *    non-overlapping runs of g tokens scored by the query of the group's last
 *    token; the pooled core tokens go through the same K/V projections as the
 *    local branch; each token sees at least its w preceding raw tokens.
 *
 * Readings taken where the pages are silent (0-indexed):
 *  - group j holds tokens [j*g, (j+1)*g - 1]; its last token is l_j = (j+1)*g - 1;
 *  - the local window of query i is [lo(i), i] with lo(i) = max(0, i - w + 1);
 *  - core j is visible to query i iff (j+1)*g <= lo(i), so n_core(i) = lo(i) / g;
 *  - pooling K and V with the group weights equals pooling the tokens and then
 *    projecting (the projection is linear and the weights sum to 1);
 *  - grouped-query attention: the pooling logit of a KV head is the mean of the
 *    logits of the r = Hq/Hkv query heads that share it, taken before the
 *    group softmax; query head h reads KV head h / r;
 *  - scale = 1/sqrt(d) unless the caller passes another; natural-log LSE.
 *
 * Variants (the ablations the pages mention; mode 0 is the method itself):
 *  - pool_mode 1, mean pooling: every token of the group weighs 1/g;
 *  - pool_mode 2, max pooling: the element-wise maximum of the group's keys
 *    and of its values (OpenReview rebuttal, pooling-ablation table);
 *  - pool_mode 3, grouped-query pooling averaged after the softmax: every
 *    query head sharing the KV head scores the group with its own last-token
 *    query and takes its own softmax; the group weights are the mean of those
 *    r weight vectors (the rebuttal leaves GQA pooling open; this is the other
 *    plain way to let r heads share one pooled K/V, and it equals pool_mode 0
 *    when r = 1);
 *  - window_mode 1, the window reaches back to the start of the group that
 *    holds lo(i): raw tokens [g*(lo(i)/g), i], so that together with the cores
 *    every earlier token is covered ("at least w preceding raw tokens").
 *
 * Layouts: Q [B, Hq, N, d], K and V [B, Hkv, N, d], Kc and Vc [B, Hkv, N/g, d],
 * O [B, Hq, N, d], LSE [B, Hq, N]; all contiguous row-major fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int64_t window_lo(int64_t i, int64_t w) { return i - w + 1 > 0 ? i - w + 1 : 0; }

int cca_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void cca_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Global-aware pooling (pooling equation): one core key and one core value per
 * (batch, KV head, group). */
void cca_oracle_pool_mode(const double *Q, const double *K, const double *V, double *Kc, double *Vc,
                          int B, int Hq, int Hkv, int N, int d, int g, double scale, int pool_mode) {
    const int64_t r = Hq / Hkv;
    const int64_t n_groups = N / g;
    const int64_t total = (int64_t)B * Hkv * n_groups;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)g);
        double *wsum = (double *)malloc(sizeof(double) * (size_t)g);
#pragma omp for schedule(static)
        for (int64_t u = 0; u < total; ++u) {
            const int64_t j = u % n_groups;
            const int64_t bk = u / n_groups; /* b * Hkv + kv head */
            const int64_t b = bk / Hkv, kv = bk % Hkv;
            const int64_t last = (j + 1) * g - 1;
            const double *Kh = K + bk * (int64_t)N * d;
            const double *Vh = V + bk * (int64_t)N * d;
            /* logits: the last token's query against every key of the group,
             * averaged over the query heads that share this KV head */
            for (int64_t t = 0; t < g; ++t) {
                const double *k = Kh + (j * g + t) * d;
                double acc = 0.0;
                for (int64_t hh = 0; hh < r; ++hh) {
                    const int64_t h = kv * r + hh;
                    const double *q = Q + ((b * Hq + h) * (int64_t)N + last) * d;
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c) dot += q[c] * k[c];
                    acc += dot;
                }
                s[t] = scale * acc / (double)r;
            }
            if (pool_mode == 3) {
                /* one softmax per query head over its own logits, then the mean of
                 * the r weight vectors weights the group's keys and values */
                for (int64_t t = 0; t < g; ++t) wsum[t] = 0.0;
                for (int64_t hh = 0; hh < r; ++hh) {
                    const int64_t h = kv * r + hh;
                    const double *q = Q + ((b * Hq + h) * (int64_t)N + last) * d;
                    for (int64_t t = 0; t < g; ++t) {
                        const double *k = Kh + (j * g + t) * d;
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += q[c] * k[c];
                        s[t] = scale * dot;
                    }
                    double hmx = s[0];
                    for (int64_t t = 1; t < g; ++t) hmx = s[t] > hmx ? s[t] : hmx;
                    double hden = 0.0;
                    for (int64_t t = 0; t < g; ++t) hden += exp(s[t] - hmx);
                    for (int64_t t = 0; t < g; ++t) wsum[t] += exp(s[t] - hmx) / hden / (double)r;
                }
                double *kc = Kc + (bk * n_groups + j) * d;
                double *vc = Vc + (bk * n_groups + j) * d;
                for (int64_t c = 0; c < d; ++c) { kc[c] = 0.0; vc[c] = 0.0; }
                for (int64_t t = 0; t < g; ++t) {
                    const double *k = Kh + (j * g + t) * d;
                    const double *v = Vh + (j * g + t) * d;
                    for (int64_t c = 0; c < d; ++c) { kc[c] += wsum[t] * k[c]; vc[c] += wsum[t] * v[c]; }
                }
                continue;
            }
            if (pool_mode == 1)
                for (int64_t t = 0; t < g; ++t) s[t] = 0.0; /* mean pooling: equal weights */
            if (pool_mode == 2) {
                /* max pooling: element-wise maximum of the group's keys and values */
                double *kc = Kc + (bk * n_groups + j) * d;
                double *vc = Vc + (bk * n_groups + j) * d;
                for (int64_t c = 0; c < d; ++c) {
                    double km = Kh[(j * g) * d + c], vm = Vh[(j * g) * d + c];
                    for (int64_t t = 1; t < g; ++t) {
                        const double kv_ = Kh[(j * g + t) * d + c], vv_ = Vh[(j * g + t) * d + c];
                        km = kv_ > km ? kv_ : km;
                        vm = vv_ > vm ? vv_ : vm;
                    }
                    kc[c] = km;
                    vc[c] = vm;
                }
                continue;
            }
            /* softmax over the group */
            double mx = s[0];
            for (int64_t t = 1; t < g; ++t) mx = s[t] > mx ? s[t] : mx;
            double den = 0.0;
            for (int64_t t = 0; t < g; ++t) { s[t] = exp(s[t] - mx); den += s[t]; }
            /* weighted sums of the group's keys and values */
            double *kc = Kc + (bk * n_groups + j) * d;
            double *vc = Vc + (bk * n_groups + j) * d;
            for (int64_t c = 0; c < d; ++c) { kc[c] = 0.0; vc[c] = 0.0; }
            for (int64_t t = 0; t < g; ++t) {
                const double a = s[t] / den;
                const double *k = Kh + (j * g + t) * d;
                const double *v = Vh + (j * g + t) * d;
                for (int64_t c = 0; c < d; ++c) { kc[c] += a * k[c]; vc[c] += a * v[c]; }
            }
        }
        free(s);
        free(wsum);
    }
}

/* Fusion equation for one query row: one softmax over the visible core tokens
 * followed by the raw tokens of the local window. */
static void attend_row(const double *q, const double *Kh, const double *Vh, const double *Kch,
                       const double *Vch, int64_t i, int64_t d, int64_t g, int64_t w, double scale,
                       int window_mode, double *z, double *o, double *lse) {
    const int64_t n_core = window_lo(i, w) / g;
    const int64_t lo = window_mode ? n_core * g : window_lo(i, w); /* first raw token */
    const int64_t n_loc = i - lo + 1;
    for (int64_t j = 0; j < n_core; ++j) {
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += q[c] * Kch[j * d + c];
        z[j] = scale * dot;
    }
    for (int64_t m = 0; m < n_loc; ++m) {
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += q[c] * Kh[(lo + m) * d + c];
        z[n_core + m] = scale * dot;
    }
    const int64_t n = n_core + n_loc;
    double mx = z[0];
    for (int64_t t = 1; t < n; ++t) mx = z[t] > mx ? z[t] : mx;
    double den = 0.0;
    for (int64_t t = 0; t < n; ++t) { z[t] = exp(z[t] - mx); den += z[t]; }
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < n_core; ++j) {
        const double a = z[j] / den;
        for (int64_t c = 0; c < d; ++c) o[c] += a * Vch[j * d + c];
    }
    for (int64_t m = 0; m < n_loc; ++m) {
        const double a = z[n_core + m] / den;
        for (int64_t c = 0; c < d; ++c) o[c] += a * Vh[(lo + m) * d + c];
    }
    *lse = mx + log(den);
}

/* Selected rows only: rows[3*t .. 3*t+2] = (b, h, i); outputs O[n_rows, d],
 * LSE[n_rows]. */
void cca_oracle_attn_rows_mode(const double *Q, const double *K, const double *V, const double *Kc,
                               const double *Vc, const int64_t *rows, int64_t n_rows, double *O,
                               double *LSE, int B, int Hq, int Hkv, int N, int d, int g, int w,
                               double scale, int window_mode) {
    (void)B;
    const int64_t r = Hq / Hkv;
    const int64_t n_groups = N / g;
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)(n_groups + (w < N ? w : N) + g + 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t t = 0; t < n_rows; ++t) {
            const int64_t b = rows[3 * t], h = rows[3 * t + 1], i = rows[3 * t + 2];
            const int64_t bk = b * Hkv + h / r;
            attend_row(Q + ((b * Hq + h) * (int64_t)N + i) * d, K + bk * (int64_t)N * d,
                       V + bk * (int64_t)N * d, Kc + bk * n_groups * d, Vc + bk * n_groups * d, i,
                       d, g, w, scale, window_mode, z, O + t * d, LSE + t);
        }
        free(z);
    }
}

/* Every row of every (batch, query head). */
void cca_oracle_attn_mode(const double *Q, const double *K, const double *V, const double *Kc,
                          const double *Vc, double *O, double *LSE, int B, int Hq, int Hkv, int N, int d,
                          int g, int w, double scale, int window_mode) {
    const int64_t r = Hq / Hkv;
    const int64_t n_groups = N / g;
    const int64_t total = (int64_t)B * Hq * N;
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)(n_groups + (w < N ? w : N) + g + 1));
#pragma omp for schedule(dynamic, 64)
        for (int64_t u = 0; u < total; ++u) {
            const int64_t i = u % N;
            const int64_t bh = u / N;
            const int64_t b = bh / Hq, h = bh % Hq;
            const int64_t bk = b * Hkv + h / r;
            attend_row(Q + u * d, K + bk * (int64_t)N * d, V + bk * (int64_t)N * d,
                       Kc + bk * n_groups * d, Vc + bk * n_groups * d, i, d, g, w, scale, window_mode,
                       z, O + u * d, LSE + u);
        }
        free(z);
    }
}

/* The method itself (pool_mode 0, window_mode 0). */
void cca_oracle_pool(const double *Q, const double *K, const double *V, double *Kc, double *Vc,
                     int B, int Hq, int Hkv, int N, int d, int g, double scale) {
    cca_oracle_pool_mode(Q, K, V, Kc, Vc, B, Hq, Hkv, N, d, g, scale, 0);
}
void cca_oracle_attn(const double *Q, const double *K, const double *V, const double *Kc,
                     const double *Vc, double *O, double *LSE, int B, int Hq, int Hkv, int N, int d,
                     int g, int w, double scale) {
    cca_oracle_attn_mode(Q, K, V, Kc, Vc, O, LSE, B, Hq, Hkv, N, d, g, w, scale, 0);
}
void cca_oracle_attn_rows(const double *Q, const double *K, const double *V, const double *Kc,
                          const double *Vc, const int64_t *rows, int64_t n_rows, double *O,
                          double *LSE, int B, int Hq, int Hkv, int N, int d, int g, int w,
                          double scale) {
    cca_oracle_attn_rows_mode(Q, K, V, Kc, Vc, rows, n_rows, O, LSE, B, Hq, Hkv, N, d, g, w, scale, 0);
}
