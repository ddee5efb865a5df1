/*
 * herald_oracle.c -- plain, slow, fp64 CPU statement of what the HERALD hot
 * path computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * bench's CPU-baseline leg call it; the product path never does.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * Sources (web pages on the subject):
 *  - "HERALD: High-Throughput Block Diffusion LLM Inference via CPU-GPU
 *    Cooperative KV Cache Retrieval", arXiv 2606.21633 v3, abstract:
 *    two-stage selection -- stage 1 scores ONE query merged from the current
 *    block's B queries against the FULL KV cache (B-fold cheaper), stage 2
 *    refines those candidates into the final top-K with the next block's real
 *    queries; the subset is reused over the block's denoising steps.
 *  - HERALD early abstract (mlsift.com listing): a single [MASK] query, double
 *    buffered sparse KV pools, subset reused T times.
 *  - SparDA (hyper.ai summary of arXiv 2606.04511), Method: a GQA group's
 *    target score is the SUM over the group's G heads of per-head softmax
 *    probabilities (the S_tgt formula); InfLLM-V2 keeps initial (sink) tokens
 *    and a local sliding window next to the top-k set.
 *
 * Readings where the pages are silent (plainest reading the rest supports):
 *  - merged query = arithmetic mean of the B queries, kept in full precision;
 *  - score scale 1/sqrt(d); no temperature;
 *  - stage 1 per-KV-head score s1[j] = sum_h softmax_j(l1[h, :])[j] over the
 *    whole context; stage 2 score s2[c] = sum over the B*G rows of the row
 *    softmax taken over the C candidates only;
 *  - every top-m keeps the m largest scores, lower position first on ties,
 *    and is stored in ascending position order;
 *  - sink = positions [0, S), local = [L-W, L), both clipped to [0, L) and
 *    unioned with the top-K without duplicates, ascending;
 *  - attention: each block query sees the selected context keys plus all B
 *    block keys (bidirectional inside the block), no mask; GQA head h reads
 *    KV head h / G.
 *
 * Layouts (all dense, row-major, fp64 here; the GPU side reads bf16 bytes
 * whose exact fp64 widening is what the tests pass in):
 *   q_*      [N][B][Hq][d]      k_cache, v_cache [N][Hkv][L_max][d]
 *   block_kv [N][B][Hkv][d]     cand [N][Hkv][C]   idx [N][Hkv][P]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int clamp_ctx(int ctx, int L_max) {
    if (ctx < 0) return 0;
    if (ctx > L_max) return L_max;
    return ctx;
}

/* Step 1 (HERALD v3 abstract: stage 1 uses one query per head formed from
 * the block's B queries; read as their mean):
 *   qbar[n][h][:] = (1/B) sum_b q_merge[n][b][h][:]. */
void oracle_merged_query(int N, int B, int Hq, int d, const double *q_merge,
                         double *qbar) {
    for (int n = 0; n < N; ++n)
        for (int h = 0; h < Hq; ++h)
            for (int e = 0; e < d; ++e) {
                double acc = 0.0;
                for (int b = 0; b < B; ++b)
                    acc += q_merge[(((size_t)n * B + b) * Hq + h) * d + e];
                qbar[((size_t)n * Hq + h) * d + e] = acc / (double)B;
            }
}

/* Step 2 (stage 1 over the full cache; GQA aggregation as SparDA's S_tgt):
 *   l1[n][h][j] = qbar[n][h] . k[n][h/G][j] / sqrt(d)       for j < ctx[n]
 *   lse1[n][h]  = log sum_j exp(l1[n][h][j])
 *   s1[n][g][j] = sum_{h in group g} exp(l1[n][h][j] - lse1[n][h])
 * Positions j >= ctx[n] get l1 = -inf and s1 = 0.  lse1 of an empty context
 * is -inf. */
void oracle_stage1_scores(int N, int Hq, int Hkv, int d, int L_max,
                          const int *ctx, const double *qbar,
                          const double *k_cache, double *l1, double *lse1,
                          double *s1) {
    const int G = Hq / Hkv;
    const double scale = 1.0 / sqrt((double)d);
#pragma omp parallel for schedule(dynamic)
    for (int ng = 0; ng < N * Hkv; ++ng) {
        const int n = ng / Hkv, g = ng % Hkv;
        const int L = clamp_ctx(ctx[n], L_max);
        const double *kbase = k_cache + ((size_t)n * Hkv + g) * L_max * d;
        double *s = s1 + ((size_t)n * Hkv + g) * L_max;
        for (int j = 0; j < L_max; ++j) s[j] = 0.0;
        for (int hl = 0; hl < G; ++hl) {
            const int h = g * G + hl;
            const double *qh = qbar + ((size_t)n * Hq + h) * d;
            double *lh = l1 + ((size_t)n * Hq + h) * L_max;
            double mx = -INFINITY;
            for (int j = 0; j < L_max; ++j) {
                if (j < L) {
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e) dot += qh[e] * kbase[(size_t)j * d + e];
                    lh[j] = dot * scale;
                    if (lh[j] > mx) mx = lh[j];
                } else {
                    lh[j] = -INFINITY;
                }
            }
            double lse = -INFINITY;
            if (L > 0) {
                double sum = 0.0;
                for (int j = 0; j < L; ++j) sum += exp(lh[j] - mx);
                lse = mx + log(sum);
            }
            lse1[(size_t)n * Hq + h] = lse;
            for (int j = 0; j < L; ++j) s[j] += exp(lh[j] - lse);
        }
    }
}

/* The m largest of score[0..n) ordered by (score descending, position
 * ascending); the chosen positions are written to out[] in ascending order.
 * Returns the count min(m, n).  Plain full sort. */
typedef struct { double s; int j; } scored_t;

static int cmp_desc_then_pos(const void *a, const void *b) {
    const scored_t *x = (const scored_t *)a, *y = (const scored_t *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

static int cmp_int(const void *a, const void *b) {
    const int x = *(const int *)a, y = *(const int *)b;
    return (x > y) - (x < y);
}

int oracle_top_m(int n, const double *score, int m, int *out) {
    if (m > n) m = n;
    if (m <= 0) return 0;
    scored_t *t = (scored_t *)malloc(sizeof(scored_t) * (size_t)n);
    for (int j = 0; j < n; ++j) { t[j].s = score[j]; t[j].j = j; }
    qsort(t, (size_t)n, sizeof(scored_t), cmp_desc_then_pos);
    for (int i = 0; i < m; ++i) out[i] = t[i].j;
    free(t);
    qsort(out, (size_t)m, sizeof(int), cmp_int);
    return m;
}

/* Step 3: per (n, g) the C_eff = min(C, ctx[n]) positions with the largest
 * s1, ascending.  cand slots past n_cand are -1. */
void oracle_topc(int N, int Hkv, int L_max, const int *ctx, const double *s1,
                 int C, int *cand, int *n_cand) {
#pragma omp parallel for schedule(dynamic)
    for (int ng = 0; ng < N * Hkv; ++ng) {
        const int n = ng / Hkv;
        const int L = clamp_ctx(ctx[n], L_max);
        int *c = cand + (size_t)ng * C;
        for (int i = 0; i < C; ++i) c[i] = -1;
        n_cand[ng] = oracle_top_m(L, s1 + (size_t)ng * L_max, C, c);
    }
}

/* Step 4 (HERALD v3 abstract, stage 2: the candidates are re-scored with the
 * real queries of the block they are selected for): rows r = (b, h) for the
 * B*G query rows of group g,
 *   l2[r][c] = q_block[n][b][h] . k[n][g][cand[c]] / sqrt(d)
 *   p[r][c]  = exp(l2[r][c] - log sum_{c'} exp(l2[r][c']))   (over candidates)
 *   s2[c]    = sum_r p[r][c]
 * Slots c >= n_cand get s2 = 0. */
void oracle_stage2_scores(int N, int B, int Hq, int Hkv, int d, int L_max,
                          const double *q_block, const double *k_cache,
                          const int *cand, const int *n_cand, int C,
                          double *s2) {
    const int G = Hq / Hkv;
    const double scale = 1.0 / sqrt((double)d);
#pragma omp parallel for schedule(dynamic)
    for (int ng = 0; ng < N * Hkv; ++ng) {
        const int n = ng / Hkv, g = ng % Hkv;
        const int nc = n_cand[ng];
        const int *c = cand + (size_t)ng * C;
        const double *kbase = k_cache + ((size_t)n * Hkv + g) * L_max * d;
        double *out = s2 + (size_t)ng * C;
        for (int i = 0; i < C; ++i) out[i] = 0.0;
        if (nc <= 0) continue;
        double *row = (double *)malloc(sizeof(double) * (size_t)nc);
        for (int b = 0; b < B; ++b)
            for (int hl = 0; hl < G; ++hl) {
                const int h = g * G + hl;
                const double *qr = q_block + (((size_t)n * B + b) * Hq + h) * d;
                double mx = -INFINITY;
                for (int i = 0; i < nc; ++i) {
                    const double *kr = kbase + (size_t)c[i] * d;
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e) dot += qr[e] * kr[e];
                    row[i] = dot * scale;
                    if (row[i] > mx) mx = row[i];
                }
                double sum = 0.0;
                for (int i = 0; i < nc; ++i) sum += exp(row[i] - mx);
                const double lse = mx + log(sum);
                for (int i = 0; i < nc; ++i) out[i] += exp(row[i] - lse);
            }
        free(row);
    }
}

/* Step 5: top-K_eff of s2 over the candidates (same order rule), then union
 * with sink [0, S) and local [L-W, L) clipped to [0, L), without duplicates,
 * ascending.  idx slots past n_sel are -1.  P is the row capacity of idx and
 * must be >= K + S + W. */
void oracle_select_final(int N, int Hkv, int L_max, const int *ctx,
                         const int *cand, const int *n_cand, const double *s2,
                         int C, int K, int S, int W, int P, int *idx,
                         int *n_sel) {
#pragma omp parallel for schedule(dynamic)
    for (int ng = 0; ng < N * Hkv; ++ng) {
        const int n = ng / Hkv;
        const int L = clamp_ctx(ctx[n], L_max);
        const int nc = n_cand[ng];
        int *slot = (int *)malloc(sizeof(int) * (size_t)(nc > 0 ? nc : 1));
        const int nk = oracle_top_m(nc, s2 + (size_t)ng * C, K, slot);
        unsigned char *keep = (unsigned char *)calloc((size_t)(L > 0 ? L : 1), 1);
        for (int i = 0; i < nk; ++i) keep[cand[(size_t)ng * C + slot[i]]] = 1;
        for (int j = 0; j < S && j < L; ++j) keep[j] = 1;
        for (int j = L - W; j < L; ++j)
            if (j >= 0) keep[j] = 1;
        int *o = idx + (size_t)ng * P;
        int cnt = 0;
        for (int i = 0; i < P; ++i) o[i] = -1;
        for (int j = 0; j < L; ++j)
            if (keep[j]) o[cnt++] = j;
        n_sel[ng] = cnt;
        free(keep);
        free(slot);
    }
}

/* Step 6 (denoising over the reused subset, bidirectional inside the block):
 * for every (n, b, h), keys = [k[n][g][idx[s]] for s < n_sel] followed by
 * [block_k[n][b'][g] for b' < B], values likewise;
 *   w = softmax(q[n][b][h] . keys^T * scale),  out[n][b][h] = sum w * values.
 * wsum (optional, [N][B][Hq]) receives sum(w) as computed. */
void oracle_sparse_attn(int N, int B, int Hq, int Hkv, int d, int L_max,
                        const double *q, const double *k_cache,
                        const double *v_cache, const int *idx,
                        const int *n_sel, int P, const double *block_k,
                        const double *block_v, double scale, double *out,
                        double *wsum) {
    const int G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic)
    for (int nbh = 0; nbh < N * B * Hq; ++nbh) {
        const int n = nbh / (B * Hq), b = (nbh / Hq) % B, h = nbh % Hq;
        const int g = h / G;
        const int ns = n_sel[n * Hkv + g];
        const int nk = ns + B;
        const double *qr = q + (size_t)nbh * d;
        double *a = (double *)malloc(sizeof(double) * (size_t)nk);
        const double **vr = (const double **)malloc(sizeof(double *) * (size_t)nk);
        double mx = -INFINITY;
        for (int s = 0; s < nk; ++s) {
            const double *kr;
            if (s < ns) {
                const size_t row = ((size_t)n * Hkv + g) * L_max + (size_t)idx[((size_t)n * Hkv + g) * P + s];
                kr = k_cache + row * d;
                vr[s] = v_cache + row * d;
            } else {
                const size_t row = ((size_t)n * B + (s - ns)) * Hkv + g;
                kr = block_k + row * d;
                vr[s] = block_v + row * d;
            }
            double dot = 0.0;
            for (int e = 0; e < d; ++e) dot += qr[e] * kr[e];
            a[s] = dot * scale;
            if (a[s] > mx) mx = a[s];
        }
        double sum = 0.0;
        for (int s = 0; s < nk; ++s) { a[s] = exp(a[s] - mx); sum += a[s]; }
        double *o = out + (size_t)nbh * d;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        double ws = 0.0;
        for (int s = 0; s < nk; ++s) {
            const double w = a[s] / sum;
            ws += w;
            for (int e = 0; e < d; ++e) o[e] += w * vr[s][e];
        }
        if (wsum) wsum[nbh] = ws;
        free(a);
        free((void *)vr);
    }
}

/* Step 7: dense reference -- step 6 with every cached position [0, ctx[n])
 * in place of the selected subset.  Written as its own loop so that
 * "dense equals sparse when the selection covers the context" is a real
 * check of step 5 and step 6. */
void oracle_dense_attn(int N, int B, int Hq, int Hkv, int d, int L_max,
                       const int *ctx, const double *q, const double *k_cache,
                       const double *v_cache, const double *block_k,
                       const double *block_v, double scale, double *out) {
    const int G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic)
    for (int nbh = 0; nbh < N * B * Hq; ++nbh) {
        const int n = nbh / (B * Hq), b = (nbh / Hq) % B, h = nbh % Hq;
        const int g = h / G;
        const int L = clamp_ctx(ctx[n], L_max);
        const double *qr = q + (size_t)nbh * d;
        double *o = out + (size_t)nbh * d;
        double mx = -INFINITY;
        for (int j = 0; j < L + B; ++j) {
            const double *kr = j < L
                ? k_cache + (((size_t)n * Hkv + g) * L_max + j) * d
                : block_k + (((size_t)n * B + (j - L)) * Hkv + g) * d;
            double dot = 0.0;
            for (int e = 0; e < d; ++e) dot += qr[e] * kr[e];
            if (dot * scale > mx) mx = dot * scale;
        }
        double sum = 0.0;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        for (int j = 0; j < L + B; ++j) {
            const double *kr, *vr;
            if (j < L) {
                kr = k_cache + (((size_t)n * Hkv + g) * L_max + j) * d;
                vr = v_cache + (((size_t)n * Hkv + g) * L_max + j) * d;
            } else {
                kr = block_k + (((size_t)n * B + (j - L)) * Hkv + g) * d;
                vr = block_v + (((size_t)n * B + (j - L)) * Hkv + g) * d;
            }
            double dot = 0.0;
            for (int e = 0; e < d; ++e) dot += qr[e] * kr[e];
            const double w = exp(dot * scale - mx);
            sum += w;
            for (int e = 0; e < d; ++e) o[e] += w * vr[e];
        }
        for (int e = 0; e < d; ++e) o[e] /= sum;
    }
}

/* Step 8 (the cache grows by the decoded block): cache[n][g][ctx[n] + b] =
 * block_kv[n][b][g] for b < B, then ctx[n] = min(ctx[n] + B, L_max): the
 * context cannot grow past the cache's capacity, and rows past L_max are
 * not written. */
void oracle_append(int N, int B, int Hkv, int d, int L_max, int *ctx,
                   const double *block_k, const double *block_v,
                   double *k_cache, double *v_cache) {
    for (int n = 0; n < N; ++n) {
        for (int b = 0; b < B; ++b)
            for (int g = 0; g < Hkv; ++g) {
                const int j = ctx[n] + b;
                if (j < 0 || j >= L_max) continue;
                const size_t dst = (((size_t)n * Hkv + g) * L_max + j) * d;
                const size_t src = (((size_t)n * B + b) * Hkv + g) * d;
                memcpy(k_cache + dst, block_k + src, sizeof(double) * (size_t)d);
                memcpy(v_cache + dst, block_v + src, sizeof(double) * (size_t)d);
            }
        /* the context grows by the block, up to the cache's capacity */
        ctx[n] = ctx[n] + B < L_max ? ctx[n] + B : L_max;
    }
}
