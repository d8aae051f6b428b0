/*
 * CPU oracle for cache-aware attention in masked-autoregressive (MAR) decoding.
 *
 * TEST INFRASTRUCTURE. This file is the plain, slow, obviously correct reference
 * that the CUDA path is checked against. Only the tests, the package smoke check
 * and the benchmark's CPU-baseline leg may load it; the library never does. It
 * shares no code, header or table with the CUDA path.
 *
 * Arithmetic: inputs arrive as float (exact copies of the bf16 or fp32 values the
 * GPU reads); every sum, exponential and division is done in double with plain
 * loops in the order the definitions state. Build with -ffp-contract=off so that
 * the result does not depend on whether the host compiler fuses multiply-adds.
 *
 * Sources (web pages, cited by title and section):
 *  [M]  "MARché: Fast Masked Autoregressive Image Generation with Cache-Aware
 *       Attention", paper notes: Method/Overall Architecture; Key Designs 1-3.
 *  [R]  "MARch'e: ... Cache-Aware Attention", machine review: "What carries the
 *       argument"; "Assumptions & free parameters" (online-softmax equivalence,
 *       the paper's Appendix A).
 *  [L]  "LazyMAR: Accelerating Masked Autoregressive Models via Feature Caching",
 *       paper notes: Key Designs, Condition Cache.
 *
 * Parity pins: every function below is pinned by tests that do not re-type its
 * formula (library routines, closed forms, invariants, brute force).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Full bidirectional softmax attention.                                     */
/*                                                                           */
/* [M] Overall Architecture: the first two decoder layers (and every layer on */
/* a periodic full-refresh step, Key Design 3) run standard full attention   */
/* over all tokens, with no causal mask. For query row i:                    */
/*   s_j = scale * <q_i, k_j>,  m = max_j s_j,  l = sum_j exp(s_j - m),      */
/*   o_i = sum_j exp(s_j - m) v_j / l,  lse_i = m + log(l).                  */
/* The softmax scale is not printed on the pages; the caller passes it      */
/* (the standard transformer value is 1/sqrt(d)).                           */
/*                                                                           */
/* Q [BH, Nq, d], K and V [BH, Nk, d] (float), O [BH, Nq, d] and LSE        */
/* [BH, Nq] (double; either may be NULL).                                    */
/* ------------------------------------------------------------------------- */
static void attend_rows(int64_t Nq, int64_t Nk, int64_t d, const float *Q,
                        const float *K, const float *V, double scale, double *O,
                        double *LSE, double *s /* Nk scratch */)
{
    for (int64_t i = 0; i < Nq; ++i) {
        const float *q = Q + i * d;
        double m = -INFINITY;
        for (int64_t j = 0; j < Nk; ++j) {
            const float *k = K + j * d;
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c) dot += (double)q[c] * (double)k[c];
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < Nk; ++j) l += exp(s[j] - m);
        if (O) {
            double *o = O + i * d;
            for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
            for (int64_t j = 0; j < Nk; ++j) {
                double p = exp(s[j] - m);
                const float *v = V + j * d;
                for (int64_t c = 0; c < d; ++c) o[c] += p * (double)v[c];
            }
            for (int64_t c = 0; c < d; ++c) o[c] /= l;
        }
        if (LSE) LSE[i] = (Nk > 0) ? m + log(l) : -INFINITY;
    }
}

void oracle_full_attn(int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                      const float *Q, const float *K, const float *V,
                      double scale, double *O, double *LSE)
{
#pragma omp parallel for schedule(dynamic)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *s = (double *)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
        attend_rows(Nq, Nk, d, Q + bh * Nq * d, K + bh * Nk * d, V + bh * Nk * d,
                    scale, O ? O + bh * Nq * d : NULL, LSE ? LSE + bh * Nq : NULL, s);
        free(s);
    }
}

/* ------------------------------------------------------------------------- */
/* Active/cached partition of one batch row.                                 */
/*                                                                           */
/* [M] Overall Architecture: the tokens split into an active set (generating, */
/* just-decoded "caching" and refreshing tokens) and a cached set holding all */
/* the remaining tokens; the two are disjoint. cached[] receives the cached  */
/* positions in ascending order. Returns the number of cached positions, or  */
/* -1 if idx holds a duplicate or out-of-range position.                     */
/* ------------------------------------------------------------------------- */
static int64_t cached_positions(int64_t N, int64_t A, const int32_t *idx,
                                int64_t *cached)
{
    unsigned char *mark = (unsigned char *)calloc((size_t)(N > 0 ? N : 1), 1);
    for (int64_t a = 0; a < A; ++a) {
        int32_t p = idx[a];
        if (p < 0 || p >= N || mark[p]) { free(mark); return -1; }
        mark[p] = 1;
    }
    int64_t C = 0;
    for (int64_t j = 0; j < N; ++j)
        if (!mark[j]) cached[C++] = j;
    free(mark);
    return C;
}

/* ------------------------------------------------------------------------- */
/* Cache-aware attention, by definition.                                     */
/*                                                                           */
/* [R] What carries the argument: active queries attend over both sets;      */
/* active tokens contribute fresh K_A/V_A, cached tokens their stored K/V.   */
/* The result is softmax attention of each active query over the key list   */
/* K* = [K_A ; cache rows at cached positions] (and V* likewise): this       */
/* function builds K*, V* explicitly and calls the full-attention oracle.    */
/*                                                                           */
/* Q_A, K_A, V_A, O [B, H, A, d]; Kc, Vc [B, H, N, d]; idx [B, A] int32;    */
/* LSE [B, H, A]. Returns 0, or -1 on an invalid idx row.                    */
/* ------------------------------------------------------------------------- */
int oracle_cache_aware_concat(int64_t B, int64_t H, int64_t N, int64_t A, int64_t d,
                              const float *Q_A, const float *K_A, const float *V_A,
                              const float *Kc, const float *Vc, const int32_t *idx,
                              double scale, double *O, double *LSE)
{
    int bad = 0;
#pragma omp parallel for schedule(dynamic)
    for (int64_t b = 0; b < B; ++b) {
        int64_t *cached = (int64_t *)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
        int64_t C = cached_positions(N, A, idx + b * A, cached);
        if (C < 0) {
#pragma omp atomic write
            bad = 1;
            free(cached);
            continue;
        }
        int64_t Nk = A + C;
        float *Ks = (float *)malloc((size_t)(Nk > 0 ? Nk : 1) * d * sizeof(float));
        float *Vs = (float *)malloc((size_t)(Nk > 0 ? Nk : 1) * d * sizeof(float));
        double *s = (double *)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
        for (int64_t h = 0; h < H; ++h) {
            int64_t bh = b * H + h;
            memcpy(Ks, K_A + bh * A * d, (size_t)(A * d) * sizeof(float));
            memcpy(Vs, V_A + bh * A * d, (size_t)(A * d) * sizeof(float));
            for (int64_t c = 0; c < C; ++c) {
                memcpy(Ks + (A + c) * d, Kc + (bh * N + cached[c]) * d, (size_t)d * sizeof(float));
                memcpy(Vs + (A + c) * d, Vc + (bh * N + cached[c]) * d, (size_t)d * sizeof(float));
            }
            attend_rows(A, Nk, d, Q_A + bh * A * d, Ks, Vs, scale,
                        O ? O + bh * A * d : NULL, LSE ? LSE + bh * A : NULL, s);
        }
        free(Ks); free(Vs); free(s); free(cached);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Cache-aware attention as the paper's two paths and merge.                 */
/*                                                                           */
/* [M] Key Design 2: alpha^(A), alpha^(C), l_i = SafeOnlineSoftmax(q_i, K_A, */
/* K_C); z_i = (alpha^(A) V_A + alpha^(C) V_C) / l_i. Each path keeps its own */
/* running max and running sum; the merge rescales both to the common max:  */
/*   m = max(m_A, m_C),  l = l_A e^(m_A-m) + l_C e^(m_C-m),                  */
/*   z = (acc_A e^(m_A-m) + acc_C e^(m_C-m)) / l,                             */
/* where an empty path has m = -inf, l = 0 and contributes nothing. [R]      */
/* Assumptions: this split equals full softmax attention (the paper's        */
/* Appendix A), which the tests check against the function above.           */
/* ------------------------------------------------------------------------- */
struct partial { double m, l; double *acc; };

static void path_partial(const float *q, int64_t n, const int64_t *rows, int64_t row0,
                         const float *Kbase, const float *Vbase, int64_t d,
                         double scale, double *s, struct partial *p)
{
    /* rows == NULL: keys are Kbase rows row0 .. row0+n-1; else Kbase rows rows[0..n). */
    p->m = -INFINITY;
    p->l = 0.0;
    for (int64_t c = 0; c < d; ++c) p->acc[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        int64_t r = rows ? rows[j] : row0 + j;
        const float *k = Kbase + r * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += (double)q[c] * (double)k[c];
        s[j] = scale * dot;
        if (s[j] > p->m) p->m = s[j];
    }
    for (int64_t j = 0; j < n; ++j) {
        int64_t r = rows ? rows[j] : row0 + j;
        double e = exp(s[j] - p->m);
        const float *v = Vbase + r * d;
        p->l += e;
        for (int64_t c = 0; c < d; ++c) p->acc[c] += e * (double)v[c];
    }
}

int oracle_cache_aware_split(int64_t B, int64_t H, int64_t N, int64_t A, int64_t d,
                             const float *Q_A, const float *K_A, const float *V_A,
                             const float *Kc, const float *Vc, const int32_t *idx,
                             double scale, double *O, double *LSE)
{
    int bad = 0;
#pragma omp parallel for schedule(dynamic)
    for (int64_t b = 0; b < B; ++b) {
        int64_t *cached = (int64_t *)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
        int64_t C = cached_positions(N, A, idx + b * A, cached);
        if (C < 0) {
#pragma omp atomic write
            bad = 1;
            free(cached);
            continue;
        }
        double *s = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
        struct partial pa, pc;
        pa.acc = (double *)malloc((size_t)d * sizeof(double));
        pc.acc = (double *)malloc((size_t)d * sizeof(double));
        for (int64_t h = 0; h < H; ++h) {
            int64_t bh = b * H + h;
            for (int64_t i = 0; i < A; ++i) {
                const float *q = Q_A + (bh * A + i) * d;
                /* active path: fresh K_A, V_A of this (b, h) */
                path_partial(q, A, NULL, bh * A, K_A, V_A, d, scale, s, &pa);
                /* cached path: stored rows of this (b, h) at the cached positions */
                for (int64_t c = 0; c < C; ++c) cached[c] += bh * N;
                path_partial(q, C, cached, 0, Kc, Vc, d, scale, s, &pc);
                for (int64_t c = 0; c < C; ++c) cached[c] -= bh * N;
                /* merge */
                double m = pa.m > pc.m ? pa.m : pc.m;
                double fa = (pa.m == -INFINITY) ? 0.0 : exp(pa.m - m);
                double fc = (pc.m == -INFINITY) ? 0.0 : exp(pc.m - m);
                double l = pa.l * fa + pc.l * fc;
                if (O) {
                    double *o = O + (bh * A + i) * d;
                    for (int64_t c = 0; c < d; ++c) o[c] = (pa.acc[c] * fa + pc.acc[c] * fc) / l;
                }
                if (LSE) LSE[bh * A + i] = m + log(l);
            }
        }
        free(pa.acc); free(pc.acc); free(s); free(cached);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* KV-cache scatter and active-row gather, as byte copies.                   */
/*                                                                           */
/* [M] Key Design 2 / Overall Architecture: active tokens project fresh K/V; */
/* the stored K/V of those positions is replaced (the per-layer cache holds  */
/* every token's latest projection). Key Design 3: a full-refresh step       */
/* overwrites every row. Rows are copied bit for bit.                        */
/*                                                                           */
/* scatter: cache[b,h,idx[b,a],:] = src[b,h,a,:]   (src [B,H,A,row])         */
/* gather : dst[b,h,a,:] = full[b,h,idx[b,a],:]    (full [B,H,N,row])        */
/* row_bytes is the byte size of one row (d * element size).                */
/* ------------------------------------------------------------------------- */
void oracle_scatter_rows(int64_t B, int64_t H, int64_t N, int64_t A, int64_t row_bytes,
                         const void *src, const int32_t *idx, void *cache)
{
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t a = 0; a < A; ++a) {
                int64_t p = idx[b * A + a];
                memcpy((char *)cache + ((b * H + h) * N + p) * row_bytes,
                       (const char *)src + ((b * H + h) * A + a) * row_bytes,
                       (size_t)row_bytes);
            }
}

void oracle_gather_rows(int64_t B, int64_t H, int64_t N, int64_t A, int64_t row_bytes,
                        const void *full, const int32_t *idx, void *dst)
{
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t a = 0; a < A; ++a) {
                int64_t p = idx[b * A + a];
                memcpy((char *)dst + ((b * H + h) * A + a) * row_bytes,
                       (const char *)full + ((b * H + h) * N + p) * row_bytes,
                       (size_t)row_bytes);
            }
}

/* ------------------------------------------------------------------------- */
/* Layer-2 head-averaged relevance score.                                    */
/*                                                                           */
/* [M] Key Design 1: during layer-2 full attention, the attention weights    */
/* (post-softmax) from every generating token to every token are averaged    */
/* across heads into a global relevance score. The pages do not say whether */
/* the generating queries are summed or averaged; averaging is taken (the   */
/* ranking is the same):                                                     */
/*   score[b, j] = 1/(H*G) * sum_h sum_g softmax_j(scale <q_{h,gen_g}, k_{h,j}>) */
/* Q, K [B, H, N, d]; gen [B, G] positions; score [B, N] double.            */
/* ------------------------------------------------------------------------- */
void oracle_l2_score(int64_t B, int64_t H, int64_t N, int64_t d, int64_t G,
                     const float *Q, const float *K, const int32_t *gen,
                     double scale, double *score)
{
#pragma omp parallel for schedule(dynamic)
    for (int64_t b = 0; b < B; ++b) {
        double *s = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
        double *sc = score + b * N;
        for (int64_t j = 0; j < N; ++j) sc[j] = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            const float *Kh = K + (b * H + h) * N * d;
            for (int64_t g = 0; g < G; ++g) {
                const float *q = Q + ((b * H + h) * N + gen[b * G + g]) * d;
                double m = -INFINITY;
                for (int64_t j = 0; j < N; ++j) {
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c) dot += (double)q[c] * (double)Kh[j * d + c];
                    s[j] = scale * dot;
                    if (s[j] > m) m = s[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j < N; ++j) l += exp(s[j] - m);
                for (int64_t j = 0; j < N; ++j) sc[j] += exp(s[j] - m) / l;
            }
        }
        for (int64_t j = 0; j < N; ++j) sc[j] /= (double)(H * G);
        free(s);
    }
}

/* ------------------------------------------------------------------------- */
/* Top-K refresh selection.                                                  */
/*                                                                           */
/* [M] Key Design 1: the K tokens with the highest relevance score become   */
/* the refreshing tokens. Candidates are all positions not in exclude[b]    */
/* (the generating and just-decoded tokens, which are active anyway and     */
/* disjoint from the refresh set). Order: higher score first, equal scores  */
/* to the lower position. The chosen K positions are returned in ascending  */
/* order. A library sort (qsort) does the ordering.                          */
/* score [B, N] double, exclude [B, E], out [B, K]. Returns 0, or -1 when a */
/* row has fewer than K candidates or exclude is out of range.               */
/* ------------------------------------------------------------------------- */
struct cand { double score; int64_t pos; };

static int by_score_then_pos(const void *x, const void *y)
{
    const struct cand *a = (const struct cand *)x, *b = (const struct cand *)y;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->pos < b->pos) ? -1 : (a->pos > b->pos);
}

static int by_pos(const void *x, const void *y)
{
    int32_t a = *(const int32_t *)x, b = *(const int32_t *)y;
    return (a > b) - (a < b);
}

int oracle_topk(int64_t B, int64_t N, const double *score, int64_t E,
                const int32_t *exclude, int64_t K, int32_t *out)
{
    int bad = 0;
    for (int64_t b = 0; b < B; ++b) {
        unsigned char *ex = (unsigned char *)calloc((size_t)(N > 0 ? N : 1), 1);
        for (int64_t e = 0; e < E; ++e) {
            int32_t p = exclude[b * E + e];
            if (p < 0 || p >= N) { bad = 1; continue; }
            ex[p] = 1;
        }
        struct cand *c = (struct cand *)malloc((size_t)(N > 0 ? N : 1) * sizeof(struct cand));
        int64_t n = 0;
        for (int64_t j = 0; j < N; ++j)
            if (!ex[j]) { c[n].score = score[b * N + j]; c[n].pos = j; ++n; }
        if (n < K) {
            bad = 1;
        } else {
            qsort(c, (size_t)n, sizeof(struct cand), by_score_then_pos);
            for (int64_t k = 0; k < K; ++k) out[b * K + k] = (int32_t)c[k].pos;
            qsort(out + b * K, (size_t)K, sizeof(int32_t), by_pos);
        }
        free(c);
        free(ex);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* LazyMAR condition cache.                                                  */
/*                                                                           */
/* [L] Condition Cache: the residual between the conditional and the         */
/* unconditional output barely changes between adjacent steps, so a cached  */
/* step runs only the conditional branch and takes                          */
/*   uncond_t = cond_t - residual_{t-1};                                     */
/* a full-compute step runs both and refreshes residual = cond - uncond.    */
/* The guided output is not printed on the pages; textbook classifier-free */
/* guidance is taken: guided = uncond + w (cond - uncond).                   */
/*                                                                           */
/* mode 0 (apply):  uncond_out = cond - residual_in                         */
/* mode 1 (update): residual_out = cond - uncond_in                          */
/* guided (may be NULL) uses the step's uncond (uncond_out in mode 0).      */
/* ------------------------------------------------------------------------- */
void oracle_cfg(int mode, int64_t n, const float *cond, const float *uncond_in,
                const float *residual_in, double w, double *uncond_out,
                double *residual_out, double *guided)
{
    for (int64_t i = 0; i < n; ++i) {
        double c = cond[i];
        double u;
        if (mode == 0) {
            u = c - (double)residual_in[i];
            uncond_out[i] = u;
        } else {
            u = (double)uncond_in[i];
            residual_out[i] = c - u;
        }
        if (guided) guided[i] = u + w * (c - u);
    }
}

/* ------------------------------------------------------------------------- */
/* Token similarity between two decode steps.                                */
/*                                                                           */
/* [L] Token Cache: in the deeper layers a token whose current feature is    */
/* close, in cosine similarity, to its cached feature reuses the cached      */
/* value. [M] Figure 1 / Figures 10-11: the same cosine between the key      */
/* (value) projections of consecutive steps shows which tokens drift.       */
/* A token's feature is the concatenation over the heads: for layout         */
/* [B, H, N, d], token (b, n) has the H*d values X[b, h, n, :] for all h.   */
/*   cos = <x, y> / (|x| |y|);  both zero -> 1, one zero -> 0.               */
/* X, Y [B, H, N, d] float (bf16 inputs widened exactly), out [B, N].       */
/* ------------------------------------------------------------------------- */
void oracle_token_cosine(int64_t B, int64_t H, int64_t N, int64_t d, const float *X,
                         const float *Y, double *out)
{
    #pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t n = 0; n < N; ++n) {
            double xy = 0.0, xx = 0.0, yy = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                const float *x = X + ((b * H + h) * N + n) * d;
                const float *y = Y + ((b * H + h) * N + n) * d;
                for (int64_t i = 0; i < d; ++i) {
                    xy += (double)x[i] * (double)y[i];
                    xx += (double)x[i] * (double)x[i];
                    yy += (double)y[i] * (double)y[i];
                }
            }
            double c;
            if (xx == 0.0 && yy == 0.0) c = 1.0;
            else if (xx == 0.0 || yy == 0.0) c = 0.0;
            else c = xy / (sqrt(xx) * sqrt(yy));
            out[b * N + n] = c;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Token-cache recompute set.                                                */
/*                                                                           */
/* [L] Token Cache: tokens whose similarity to the cached feature is high   */
/* reuse the cached value; the others are recomputed. Here a token is       */
/* recomputed unless cos > tau (so a NaN similarity is recomputed), or when  */
/* it is in the forced set (e.g. the tokens decoded at this step). The       */
/* decision is taken on the given fp32 similarities.                         */
/* cos [B, N] float, force [B, F] (F may be 0), out_idx [B, N]: the          */
/* recomputed positions ascending, then -1; out_count [B].                   */
/* Returns -1 when a forced position is out of range (it is ignored).        */
/* ------------------------------------------------------------------------- */
int oracle_select_recompute(int64_t B, int64_t N, const float *cosv, float tau,
                            const int32_t *force, int64_t F, int32_t *out_idx,
                            int32_t *out_count)
{
    int bad = 0;
    for (int64_t b = 0; b < B; ++b) {
        unsigned char *f = (unsigned char *)calloc((size_t)(N > 0 ? N : 1), 1);
        for (int64_t k = 0; k < F; ++k) {
            int32_t p = force[b * F + k];
            if (p < 0 || p >= N) { bad = 1; continue; }
            f[p] = 1;
        }
        int32_t cnt = 0;
        for (int64_t n = 0; n < N; ++n) {
            const float c = cosv[b * N + n];
            if (f[n] || !(c > tau)) out_idx[b * N + cnt++] = (int32_t)n;
        }
        for (int64_t n = cnt; n < N; ++n) out_idx[b * N + n] = -1;
        out_count[b] = cnt;
        free(f);
    }
    return bad ? -1 : 0;
}
