/*
 * rpe_oracle.c -- the oracle for relative-position attention on a 2D patch grid.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test suite, the smoke check
 * and the benchmark's CPU-baseline / reference arm load this file. The CUDA
 * library never includes, links or calls it, and it shares no header, helper
 * or constant with that library.
 *
 * Everything here is the plain definition, evaluated pair by pair in double
 * precision with no blocking, fusion or reordering beyond what the pages
 * state. Sources (page title, then the section or equation on it):
 *
 *   [iRPE]  "Rethinking and Improving Relative Position Encoding for Vision
 *           Transformer" (summary card): Method, eqs. 13-18, 25-28; the
 *           Pitfalls list; the Paper-vs-code list.
 *   [SWIN2D] "Swin 的二维 RPE" (Deep-learning notes 24, Swin's 2D RPE):
 *           sections 2.2, 3.1, 3.2 (worked example, M = 3), 3.3.
 *   [SWIN]  "Swin Transformer, section 3.2 and Table 4" (SOTA practice record):
 *           Attention(Q,K,V) = SoftMax(Q K^T / sqrt(d) + B) V.
 *   [SHAW]  "Implementation: Relative Position in Self-Attention": the
 *           embedding table section (clip and shift to [0, 2k]) and the
 *           score / output sections (per-pair double loop).
 *
 * Readings taken where the pages are silent:
 *   - offsets are query minus key in 2D (the SWIN2D worked example: patch
 *     (0,0) attending (2,2) gives (-2,-2));
 *   - the row offset is the major index of a Product id and of a Swin index;
 *   - Python round() is round-half-to-even, reproduced with nearbyint();
 *   - contextual key and query terms sit inside the 1/sqrt(d) scaling, the
 *     Swin bias is added after it;
 *   - the value term uses the post-softmax weights and the same bucket ids.
 *
 * Every function here is pinned by a CPU test (tests/test_oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_K 1u /* contextual term on keys    (iRPE eq. 15) */
#define ORC_Q 2u /* contextual term on queries (iRPE eq. 16) */
#define ORC_V 4u /* contextual term on values  (iRPE eq. 17) */

/* ---------------------------------------------------------------------- */
/* Index functions                                                        */
/* ---------------------------------------------------------------------- */

/* iRPE eq. 18, the piecewise index g(x) of one axis offset.
 * |x| <= alpha: the offset itself, rounded.
 * otherwise:    log-spaced between alpha and gamma, scaled into
 *               [alpha, beta], rounded, capped at beta, then truncated
 *               toward zero after the sign is applied (Paper-vs-code list:
 *               the code truncates toward zero). */
int orc_piecewise_index(double x, double alpha, double beta, double gamma)
{
    if (fabs(x) <= alpha)
        return (int)nearbyint(x);
    double log_share = log(fabs(x) / alpha) / log(gamma / alpha);
    double spread = alpha + log_share * (beta - alpha);
    double rounded = nearbyint(spread);
    double capped = (beta < rounded) ? beta : rounded;
    double sign = (x > 0.0) ? 1.0 : -1.0;
    return (int)(sign * capped);
}

/* iRPE eq. 25 (Product mapping) on an H x W grid, tokens in row-major order.
 * Writes ids[i*N + j] for query i and key j, N = H*W. The table half-width
 * is int(beta) (Pitfalls: "use int(beta) for the table size"), so ids lie
 * in [0, (2*int(beta)+1)^2). Returns the number of buckets. */
/* One query row of the Product map: ids_i[j] for query i and every key j. */
static void product_ids_row(int H, int W, double alpha, double beta, double gamma, int i,
                            int32_t *ids_i)
{
    int half = (int)beta;
    int span = 2 * half + 1;
    int ri = i / W, ci = i % W;
    for (int j = 0; j < H * W; ++j) {
        int rj = j / W, cj = j % W;
        int row_index = orc_piecewise_index((double)(ri - rj), alpha, beta, gamma);
        int col_index = orc_piecewise_index((double)(ci - cj), alpha, beta, gamma);
        ids_i[j] = (row_index + half) * span + (col_index + half);
    }
}

int orc_product_bucket_ids(int H, int W, double alpha, double beta, double gamma,
                           int32_t *ids)
{
    int span = 2 * (int)beta + 1;
    int N = H * W;
    for (int i = 0; i < N; ++i)
        product_ids_row(H, W, alpha, beta, gamma, i, ids + (int64_t)i * N);
    return span * span;
}

/* iRPE section 3.2, Euclidean mapping (undirected): the bucket comes from the
 * Euclidean length of the 2D offset through the same index function. The
 * distance is rounded before the index (the Paper-vs-code list: the code
 * rounds first; round half to even, as Python does). The table has
 * 2*int(beta)+1 entries (section 3.2: 2 beta + 1 buckets); the index, in
 * [0, int(beta)] for a distance, is stored shifted by int(beta), the same
 * shift as one axis of a directed mapping. Writes ids[i*N + j]; returns the
 * number of buckets. */
int orc_euclidean_bucket_ids(int H, int W, double alpha, double beta, double gamma,
                             int32_t *ids)
{
    int half = (int)beta;
    int N = H * W;
    for (int i = 0; i < N; ++i) {
        int ri = i / W, ci = i % W;
        for (int j = 0; j < N; ++j) {
            int dr = ri - j / W, dc = ci - j % W;
            double dist = nearbyint(sqrt((double)dr * dr + (double)dc * dc));
            ids[(int64_t)i * N + j] = orc_piecewise_index(dist, alpha, beta, gamma) + half;
        }
    }
    return 2 * half + 1;
}

/* iRPE section 3.2, Cross mapping (directed; eqs. 22-24): one bucket for the
 * row offset and one for the column offset, each through the index function,
 * with their two encodings added. The table has 2 * (2*int(beta)+1) entries
 * (section 3.2: 2 x (2 beta + 1) buckets): row buckets first, then column
 * buckets. Writes ids_row[i*N + j] in [0, span) and ids_col[i*N + j] in
 * [span, 2*span), span = 2*int(beta)+1; returns 2*span. */
int orc_cross_bucket_ids(int H, int W, double alpha, double beta, double gamma,
                         int32_t *ids_row, int32_t *ids_col)
{
    int half = (int)beta;
    int span = 2 * half + 1;
    int N = H * W;
    for (int i = 0; i < N; ++i) {
        int ri = i / W, ci = i % W;
        for (int j = 0; j < N; ++j) {
            int rj = j / W, cj = j % W;
            ids_row[(int64_t)i * N + j] = orc_piecewise_index((double)(ri - rj), alpha, beta, gamma) + half;
            ids_col[(int64_t)i * N + j] = span + orc_piecewise_index((double)(ci - cj), alpha, beta, gamma) + half;
        }
    }
    return 2 * span;
}

/* The clip index as a 2D index function (iRPE table 3, "clip versus
 * piecewise"; the clip of SHAW's embedding-table section): each axis offset,
 * query minus key as for the piecewise index, is clipped to [-k, k], and the
 * two clipped offsets form a Product id (eq. 25) over (2k+1)^2 buckets.
 * Writes ids[i*N + j]; returns (2k+1)^2. */
int orc_clip_product_bucket_ids(int H, int W, int k, int32_t *ids)
{
    int span = 2 * k + 1;
    int N = H * W;
    for (int i = 0; i < N; ++i) {
        int ri = i / W, ci = i % W;
        for (int j = 0; j < N; ++j) {
            int dr = ri - j / W, dc = ci - j % W;
            if (dr < -k) dr = -k;
            if (dr > k) dr = k;
            if (dc < -k) dc = -k;
            if (dc > k) dc = k;
            ids[(int64_t)i * N + j] = (dr + k) * span + (dc + k);
        }
    }
    return span * span;
}

/* iRPE section 4.1: the class token gets one extra bucket for all its
 * pairs. Token 0 is the class token and tokens 1..N the patches (patch t at
 * grid token t - 1). Given the patches' id map ids [N, N] of K buckets,
 * writes the (N+1) x (N+1) map out with bucket K on row 0 and column 0 and
 * ids[i-1][j-1] elsewhere. Returns K + 1. */
int orc_add_cls_bucket(int N, const int32_t *ids, int K, int32_t *out)
{
    int n = N + 1;
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j)
            out[(int64_t)i * n + j] = (i == 0 || j == 0) ? K : ids[(int64_t)(i - 1) * N + (j - 1)];
    return K + 1;
}

/* SWIN2D sections 3.1-3.2: inside an M x M window the offsets lie in
 * [-(M-1), M-1]; shifting by M-1 moves them to [0, 2M-2]; the compact
 * (2M-1) x (2M-1) table is read at (dr', dc') and, flattened to 1D, at
 * dr' * (2M-1) + dc'. Writes idx[i*n + j], n = M*M. Returns (2M-1)^2. */
int orc_swin_bias_index(int M, int32_t *idx)
{
    int n = M * M;
    int side = 2 * M - 1;
    for (int i = 0; i < n; ++i) {
        int ri = i / M, ci = i % M;
        for (int j = 0; j < n; ++j) {
            int rj = j / M, cj = j % M;
            int dr = ri - rj + (M - 1);
            int dc = ci - cj + (M - 1);
            idx[i * n + j] = dr * side + dc;
        }
    }
    return side * side;
}

/* SHAW, embedding-table section: a 1D offset j - i is clipped to [-k, k]
 * and shifted by k into an index in [0, 2k]. Writes ids[i*n + j]. */
void orc_clip_ids_1d(int n, int k, int32_t *ids)
{
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) {
            int rel = j - i;
            if (rel < -k) rel = -k;
            if (rel > k) rel = k;
            ids[i * n + j] = rel + k;
        }
}

/* ---------------------------------------------------------------------- */
/* Attention with a relative term, per pair                               */
/* ---------------------------------------------------------------------- */

static double dot(const double *a, const double *b, int d)
{
    double s = 0.0;
    for (int c = 0; c < d; ++c)
        s += a[c] * b[c];
    return s;
}

/* One (batch, head) slice of n tokens with head dim d, everything per pair:
 *
 *   e_ij = ( q_i.k_j                      content term       (iRPE eq. 13)
 *          + [tab_k] q_i . tab_k[id_ij]   contextual key     (iRPE eq. 15)
 *          + [tab_q] k_j . tab_q[id_ij]   contextual query   (iRPE eq. 16)
 *          + [bias_in] bias_in[id_ij] )   bias mode: a scalar per bucket,
 *                                         inside the scaling  (iRPE eqs. 13-14)
 *          * scale
 *          + [bias] bias[id_ij]           Swin bias, after the scaling (SWIN)
 *   a_ij = exp(e_ij - max_j e_ij) / sum_j exp(e_ij - max_j e_ij)
 *   z_i  = sum_j a_ij v_j + [tab_v] sum_j a_ij tab_v[id_ij]   (iRPE eq. 17)
 *
 * ids is n x n (query-major); tables are [num_buckets x d]; bias and bias_in
 * have one scalar per bucket. ids2, when not NULL, is a second n x n id map
 * whose entries of every iRPE term (tab_k, tab_q, tab_v, bias_in) are added
 * to those of ids: the Cross mapping's column buckets (iRPE eqs. 22-24). Any of tab_k, tab_q, tab_v, bias, bias_in may be
 * NULL (term off).
 * rows lists the query rows to compute (NULL: all n); out and attn are
 * written only at those rows. attn may be NULL. Returns 0, or -1 on a bad id. */
/* One query row of orc_attention: query qi against every key, its ids ids_i[j]
 * (and ids2_i, or NULL) for key j; e is scratch of n doubles; zi receives the
 * d outputs and attn_i (or NULL) the n weights. Returns 0, or -1 on a bad id. */
static int attention_row(int n, int d, const double *qi, const double *k, const double *v,
                         const int32_t *ids_i, const int32_t *ids2_i, int num_buckets,
                         const double *tab_k, const double *tab_q, const double *tab_v,
                         const double *bias, const double *bias_in, double scale,
                         double *e, double *zi, double *attn_i)
{
    double emax = -INFINITY;
    for (int j = 0; j < n; ++j) {
        int id = ids_i[j];
        if (id < 0 || id >= num_buckets) return -1;
        int id2 = ids2_i ? ids2_i[j] : -1;
        if (ids2_i && (id2 < 0 || id2 >= num_buckets)) return -1;
        const double *kj = k + (int64_t)j * d;
        double logit = dot(qi, kj, d);
        if (tab_k) logit += dot(qi, tab_k + (int64_t)id * d, d);
        if (tab_q) logit += dot(kj, tab_q + (int64_t)id * d, d);
        if (bias_in) logit += bias_in[id];
        if (ids2_i) {
            if (tab_k) logit += dot(qi, tab_k + (int64_t)id2 * d, d);
            if (tab_q) logit += dot(kj, tab_q + (int64_t)id2 * d, d);
            if (bias_in) logit += bias_in[id2];
        }
        logit *= scale;
        if (bias) logit += bias[id];
        e[j] = logit;
        if (logit > emax) emax = logit;
    }
    double denom = 0.0;
    for (int j = 0; j < n; ++j) {
        e[j] = exp(e[j] - emax);
        denom += e[j];
    }
    for (int c = 0; c < d; ++c) zi[c] = 0.0;
    for (int j = 0; j < n; ++j) {
        double a = e[j] / denom;
        if (attn_i) attn_i[j] = a;
        const double *vj = v + (int64_t)j * d;
        for (int c = 0; c < d; ++c) zi[c] += a * vj[c];
        if (tab_v) {
            const double *rv = tab_v + (int64_t)ids_i[j] * d;
            for (int c = 0; c < d; ++c) zi[c] += a * rv[c];
            if (ids2_i) {
                rv = tab_v + (int64_t)ids2_i[j] * d;
                for (int c = 0; c < d; ++c) zi[c] += a * rv[c];
            }
        }
    }
    return 0;
}

int orc_attention(int n, int d, const double *q, const double *k, const double *v,
                  const int32_t *ids, const int32_t *ids2, int num_buckets,
                  const double *tab_k, const double *tab_q, const double *tab_v,
                  const double *bias, const double *bias_in, double scale,
                  int nrows, const int32_t *rows, double *out, double *attn)
{
    double *e = (double *)malloc(sizeof(double) * (size_t)n);
    if (!e) return -2;
    int count = rows ? nrows : n;
    int status = 0;
    for (int r = 0; r < count && status == 0; ++r) {
        int64_t i = rows ? rows[r] : r;
        status = attention_row(n, d, q + i * d, k, v, ids + i * n, ids2 ? ids2 + i * n : NULL,
                               num_buckets, tab_k, tab_q, tab_v, bias, bias_in, scale, e,
                               out + i * d, attn ? attn + i * n : NULL);
    }
    free(e);
    return status;
}

/* The same slice by the efficient route of iRPE section 3.2 (eqs. 26-28):
 * every query is dotted with every bucket vector once (QR = q tab_k^T, n x K),
 * every key with every query-side bucket vector (KR = k tab_q^T), and the
 * n x n position terms are gathers from those by bucket id. The value term
 * sums the weights per bucket first (PB, n x K) and multiplies by tab_v once.
 * It exists only so a test can check that it equals orc_attention. */
int orc_attention_efficient(int n, int d, const double *q, const double *k, const double *v,
                            const int32_t *ids, int num_buckets,
                            const double *tab_k, const double *tab_q, const double *tab_v,
                            const double *bias, double scale, double *out)
{
    int K = num_buckets;
    double *qr = (double *)calloc((size_t)n * K, sizeof(double));
    double *kr = (double *)calloc((size_t)n * K, sizeof(double));
    double *pb = (double *)calloc((size_t)K, sizeof(double));
    double *e = (double *)malloc(sizeof(double) * (size_t)n);
    if (!qr || !kr || !pb || !e) { free(qr); free(kr); free(pb); free(e); return -2; }
    for (int i = 0; i < n; ++i)
        for (int b = 0; b < K; ++b) {
            if (tab_k) qr[(int64_t)i * K + b] = dot(q + (int64_t)i * d, tab_k + (int64_t)b * d, d);
            if (tab_q) kr[(int64_t)i * K + b] = dot(k + (int64_t)i * d, tab_q + (int64_t)b * d, d);
        }
    int status = 0;
    for (int i = 0; i < n && status == 0; ++i) {
        double emax = -INFINITY;
        for (int j = 0; j < n; ++j) {
            int id = ids[(int64_t)i * n + j];
            if (id < 0 || id >= K) { status = -1; break; }
            double logit = dot(q + (int64_t)i * d, k + (int64_t)j * d, d)
                         + qr[(int64_t)i * K + id] + kr[(int64_t)j * K + id];
            logit = logit * scale + (bias ? bias[id] : 0.0);
            e[j] = logit;
            if (logit > emax) emax = logit;
        }
        if (status) break;
        double denom = 0.0;
        for (int j = 0; j < n; ++j) { e[j] = exp(e[j] - emax); denom += e[j]; }
        for (int b = 0; b < K; ++b) pb[b] = 0.0;
        double *zi = out + (int64_t)i * d;
        for (int c = 0; c < d; ++c) zi[c] = 0.0;
        for (int j = 0; j < n; ++j) {
            double a = e[j] / denom;
            pb[ids[(int64_t)i * n + j]] += a;
            for (int c = 0; c < d; ++c) zi[c] += a * v[(int64_t)j * d + c];
        }
        if (tab_v)
            for (int b = 0; b < K; ++b)
                for (int c = 0; c < d; ++c) zi[c] += pb[b] * tab_v[(int64_t)b * d + c];
    }
    free(qr); free(kr); free(pb); free(e);
    return status;
}

/* ---------------------------------------------------------------------- */
/* Whole-tensor forms of the two workloads                                */
/* ---------------------------------------------------------------------- */

/* iRPE contextual Product attention over q, k, v of shape [B, heads, N, d],
 * N = H*W, with head-shared tables [num_buckets, d] selected by flags
 * (ORC_K | ORC_Q | ORC_V). Bucket ids are built here from the definition, for
 * the listed query rows only (no N x N map when rows are given).
 * slice_list / nslices pick (b*heads + h) slices (NULL: all) and rows /
 * nrows pick query rows within each (NULL: all). Returns 0 on success. */
int orc_irpe_attention(int B, int heads, int H, int W, int d,
                       double alpha, double beta, double gamma, unsigned flags,
                       const double *q, const double *k, const double *v,
                       const double *tab_q, const double *tab_k, const double *tab_v,
                       int nslices, const int32_t *slice_list,
                       int nrows, const int32_t *rows, double *out)
{
    int N = H * W;
    /* the id rows of the listed queries only (all N when rows is NULL) */
    int count_rows = rows ? nrows : N;
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * ((size_t)count_rows * N + 1));
    double *e = (double *)malloc(sizeof(double) * (size_t)N);
    if (!ids || !e) { free(ids); free(e); return -2; }
    for (int r = 0; r < count_rows; ++r)
        product_ids_row(H, W, alpha, beta, gamma, rows ? rows[r] : r, ids + (int64_t)r * N);
    int K = (2 * (int)beta + 1) * (2 * (int)beta + 1);
    double scale = 1.0 / sqrt((double)d);
    int count = slice_list ? nslices : B * heads;
    int status = 0;
    for (int s = 0; s < count && status == 0; ++s) {
        int64_t bh = slice_list ? slice_list[s] : s;
        int64_t off = bh * (int64_t)N * d;
        for (int r = 0; r < count_rows && status == 0; ++r) {
            int64_t i = rows ? rows[r] : r;
            status = attention_row(N, d, q + off + i * d, k + off, v + off, ids + (int64_t)r * N,
                                   NULL, K, (flags & ORC_K) ? tab_k : NULL,
                                   (flags & ORC_Q) ? tab_q : NULL, (flags & ORC_V) ? tab_v : NULL,
                                   NULL, NULL, scale, e, out + off + i * d, NULL);
        }
    }
    free(ids);
    free(e);
    return status;
}

/* iRPE attention over q, k, v [B, heads, N, d] with a caller-given id map
 * ids [N, N] of num_buckets buckets (any mapping: Product, Euclidean, ...),
 * an optional second map ids2 [N, N] whose entries are added (Cross),
 * contextual tables [tab_heads, num_buckets, d] (tab_heads 1: one table shared
 * by every head; else one per head, head h reading table h; iRPE section 4.2,
 * table 2: shared or separate per head),
 * head-shared contextual tables selected by flags, and an optional bias-mode
 * table bias_in [num_buckets, bias_heads] (iRPE eq. 14; bias_heads is 1 for
 * one table shared by every head, else heads; column h serves head h).
 * slice_list / rows as for orc_irpe_attention. */
int orc_irpe_attention_ids(int B, int heads, int N, int d, const int32_t *ids,
                           const int32_t *ids2, int num_buckets, unsigned flags,
                           const double *q, const double *k, const double *v,
                           const double *tab_q, const double *tab_k, const double *tab_v,
                           int tab_heads, const double *bias_in, int bias_heads,
                           int nslices, const int32_t *slice_list,
                           int nrows, const int32_t *rows, double *out)
{
    double *bias = NULL;
    if (bias_in) {
        bias = (double *)malloc(sizeof(double) * (size_t)num_buckets);
        if (!bias) return -2;
    }
    double scale = 1.0 / sqrt((double)d);
    int count = slice_list ? nslices : B * heads;
    int status = 0;
    for (int s = 0; s < count && status == 0; ++s) {
        int64_t bh = slice_list ? slice_list[s] : s;
        if (bias_in) {
            int h = bias_heads == 1 ? 0 : (int)(bh % heads);
            for (int b = 0; b < num_buckets; ++b) bias[b] = bias_in[(int64_t)b * bias_heads + h];
        }
        int64_t off = bh * (int64_t)N * d;
        int64_t toff = tab_heads == 1 ? 0 : (bh % heads) * (int64_t)num_buckets * d;
        status = orc_attention(N, d, q + off, k + off, v + off, ids, ids2, num_buckets,
                               (flags & ORC_K) ? tab_k + toff : NULL,
                               (flags & ORC_Q) ? tab_q + toff : NULL,
                               (flags & ORC_V) ? tab_v + toff : NULL,
                               NULL, bias, scale, nrows, rows, out + off, NULL);
    }
    free(bias);
    return status;
}

/* Swin window attention (SWIN; SWIN2D section 3.2) over q, k, v of shape
 * [num_windows, heads, M*M, d] with the compact table laid out
 * [(2M-1)^2, heads] (bucket-major, one column per head). */
int orc_swin_attention(int num_windows, int heads, int M, int d,
                       const double *q, const double *k, const double *v,
                       const double *table, int nslices, const int32_t *slice_list,
                       double *out)
{
    int n = M * M;
    int nb = (2 * M - 1) * (2 * M - 1);
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)n * n);
    double *bias = (double *)malloc(sizeof(double) * (size_t)nb);
    if (!idx || !bias) { free(idx); free(bias); return -2; }
    orc_swin_bias_index(M, idx);
    double scale = 1.0 / sqrt((double)d);
    int count = slice_list ? nslices : num_windows * heads;
    int status = 0;
    for (int s = 0; s < count && status == 0; ++s) {
        int64_t wh = slice_list ? slice_list[s] : s;
        int h = (int)(wh % heads);
        for (int b = 0; b < nb; ++b) bias[b] = table[(int64_t)b * heads + h];
        int64_t off = wh * (int64_t)n * d;
        status = orc_attention(n, d, q + off, k + off, v + off, idx, NULL, nb,
                               NULL, NULL, NULL, bias, NULL, scale, 0, NULL, out + off, NULL);
    }
    free(idx); free(bias);
    return status;
}
