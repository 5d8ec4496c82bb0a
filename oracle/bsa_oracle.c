/*
 * bsa_oracle.c -- plain, slow, obviously-correct CPU oracle for block-sparse
 * attention with a mean-pooled top-k block selector.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this library. The product path
 * (the CUDA library) never calls it, and the two share no code.
 *
 * Sources (page title, section):
 *   [P1] "多模态DiT中的块稀疏注意力：从原理到工程落地"
 *        §2.1 block mask: a block pair is computed whole or skipped whole;
 *        §3.1-§3.2 modality regions, image local band + global anchors,
 *        video cuboids decided by 3-D coordinates;
 *        §4.1 the block-sparse FlashAttention loop over active_kv_blocks[i],
 *        index kept in device memory as CSR or a bitmap tested by popcount;
 *        §4.3 skipped blocks count as score -inf, normaliser is the true sum.
 *   [P3] "Can sparse attention close the quality gap in diffusion
 *        transformers", section on mean-pooled block scoring: naive BSA scores
 *        each (Q block, KV block) pair by the dot product of the mean-pooled
 *        query and key block representations and keeps the top-scoring KV
 *        blocks at the given density.
 *
 * Readings where the pages leave a step open (all stated, none invented):
 *   R1 pooling: each element taken exactly as fp32, summed over the block's
 *      tokens t = 0..bs-1 in order in fp32 round-to-nearest, no contraction,
 *      then multiplied by 1/bs (a power of two, exact).
 *   R2 score: acc = +0; for c = 0..d-1: acc = fmaf(qbar[c], kbar[c], acc).
 *      No 1/sqrt(d) and no softmax: both are monotone and leave the ranking.
 *   R3 top-k: k = max(1, floor(density * nKB)) with density taken as float32
 *      and the product in double (P1 §5.3 asks for a per-Q-block target
 *      count). Order: value descending with -0 == +0, equal values -> lower
 *      block index first. A NaN score is an error.
 *   R4 attention: s_rc = scale * q_r.k_c for keys c in active blocks of the
 *      row's Q block, -inf otherwise; O_r = sum_c softmax(s_r)_c v_c,
 *      LSE_r = ln sum_c exp(s_rc). Computed as the definition: full score
 *      row, two passes (max, then sum). Inputs upcast exactly to double.
 *   R5 empty active set: O_r = 0, LSE_r = -inf (the definition gives 0/0).
 *
 * Parity pins (tests/test_oracle_pins.py) tie every function here to closed
 * forms, brute force or library routines; no function is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NONFINITE 5

/* ---------------------------------------------------------------------- */
/* [P3] naive BSA step 1: mean-pooled block representation (reading R1):  */
/* the mean of the block's tokens; a ragged last block (N not a multiple   */
/* of bs, reading R20) averages the tokens it holds.                       */
/* X: [n_heads][N][d] fp32; out: [n_heads][ceil(N/bs)][d] fp32.            */
int bsa_oracle_block_mean(const float *X, int64_t n_heads, int64_t N, int d, int bs,
                          float *out)
{
    if (!X || !out || n_heads <= 0 || N <= 0 || d <= 0 || bs <= 0)
        return ORACLE_ERR_ARG;
    const int64_t nB = (N + bs - 1) / bs;
    for (int64_t h = 0; h < n_heads; ++h)
        for (int64_t i = 0; i < nB; ++i) {
            const int64_t cnt = (N - i * bs) < bs ? (N - i * bs) : bs;
            for (int c = 0; c < d; ++c) {
                float acc = 0.0f;
                for (int64_t t = 0; t < cnt; ++t)
                    acc = acc + X[(h * N + i * bs + t) * d + c];
                out[(h * nB + i) * d + c] = acc / (float)cnt;
            }
        }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* [P3] naive BSA step 2: score of each (Q block, KV block) pair is the   */
/* dot product of the pooled representations (reading R2).               */
/* qbar: [n_heads][nQB][d], kbar: [n_heads][nKB][d], scores: [n_heads][nQB][nKB] */
int bsa_oracle_block_scores(const float *qbar, const float *kbar, int64_t n_heads, int nQB,
                            int nKB, int d, float *scores)
{
    if (!qbar || !kbar || !scores || n_heads <= 0 || nQB <= 0 || nKB <= 0 || d <= 0)
        return ORACLE_ERR_ARG;
    for (int64_t h = 0; h < n_heads; ++h)
        for (int i = 0; i < nQB; ++i)
            for (int j = 0; j < nKB; ++j) {
                const float *a = qbar + (h * nQB + i) * d;
                const float *b = kbar + (h * nKB + j) * d;
                float acc = 0.0f;
                for (int c = 0; c < d; ++c)
                    acc = fmaf(a[c], b[c], acc);
                scores[(h * nQB + i) * (int64_t)nKB + j] = acc;
            }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* [P3] naive BSA step 3 / [P1] §5.3 per-Q-block target count (reading R3). */
int bsa_oracle_topk_count(float density, int nKB)
{
    int k = (int)floor((double)density * (double)nKB);
    if (k < 1) k = 1;
    if (k > nKB) k = nKB;
    return k;
}

static const float *g_row; /* qsort comparator context (single-threaded use) */

static int cmp_score_desc_index_asc(const void *pa, const void *pb)
{
    int a = *(const int *)pa, b = *(const int *)pb;
    float va = g_row[a], vb = g_row[b]; /* -0 == +0 under C comparison */
    if (va > vb) return -1;
    if (va < vb) return 1;
    return (a < b) ? -1 : (a > b) ? 1 : 0;
}

/* scores: [n_rows][nKB]; mask: [n_rows][nKB] (1 = kept). */
int bsa_oracle_topk(const float *scores, int64_t n_rows, int nKB, int k, uint8_t *mask)
{
    if (!scores || !mask || n_rows <= 0 || nKB <= 0 || k < 1 || k > nKB) return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < n_rows * nKB; ++r)
        if (isnan(scores[r])) return ORACLE_ERR_NONFINITE;
    int *order = (int *)malloc(sizeof(int) * (size_t)nKB);
    if (!order) return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < n_rows; ++r) {
        g_row = scores + r * nKB;
        for (int j = 0; j < nKB; ++j) order[j] = j;
        qsort(order, (size_t)nKB, sizeof(int), cmp_score_desc_index_asc);
        memset(mask + r * nKB, 0, (size_t)nKB);
        for (int t = 0; t < k; ++t) mask[r * nKB + order[t]] = 1;
    }
    free(order);
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* [P1] §3.1-§3.2 static text + image mask: leading text blocks are dense  */
/* in both directions; image blocks form a local band |r-c| <= band plus   */
/* global anchor blocks that are dense in both directions.                */
/* mask: [nB][nB].                                                         */
int bsa_oracle_band_mask(int nB, int n_text, int band, const int *anchors, int n_anchors,
                         uint8_t *mask)
{
    if (!mask || nB <= 0 || n_text < 0 || n_text > nB || band < 0 || n_anchors < 0)
        return ORACLE_ERR_ARG;
    for (int i = 0; i < nB; ++i)
        for (int j = 0; j < nB; ++j) {
            int on = 0;
            if (i < n_text || j < n_text) {
                on = 1;
            } else {
                int r = i - n_text, c = j - n_text;
                if (abs(r - c) <= band) on = 1;
                for (int a = 0; a < n_anchors; ++a)
                    if (r == anchors[a] || c == anchors[a]) on = 1;
            }
            mask[(int64_t)i * nB + j] = (uint8_t)on;
        }
    return ORACLE_OK;
}

/* [P1] §3.2 video cuboid attention: leading text blocks dense both ways; */
/* cuboid blocks (t-major raster over a gt x gh x gw grid) attend to their */
/* own cuboid and the face-adjacent ones (6-neighbourhood, clipped).       */
int bsa_oracle_cuboid_mask(int n_text, int gt, int gh, int gw, uint8_t *mask)
{
    if (!mask || n_text < 0 || gt <= 0 || gh <= 0 || gw <= 0) return ORACLE_ERR_ARG;
    const int nB = n_text + gt * gh * gw;
    for (int i = 0; i < nB; ++i)
        for (int j = 0; j < nB; ++j) {
            int on = 0;
            if (i < n_text || j < n_text) {
                on = 1;
            } else {
                int a = i - n_text, b = j - n_text;
                int at = a / (gh * gw), ah = (a / gw) % gh, aw = a % gw;
                int bt = b / (gh * gw), bh = (b / gw) % gh, bw = b % gw;
                int dist = abs(at - bt) + abs(ah - bh) + abs(aw - bw);
                on = (dist <= 1);
            }
            mask[(int64_t)i * nB + j] = (uint8_t)on;
        }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* [P1] §4.1 index forms: active_kv_blocks[i] as CSR (row_ptr, col_idx     */
/* ascending) and as a bitmap with one bit per block (bit j%32 of word     */
/* j/32). Returns nnz, or -1 on bad arguments.                             */
int64_t bsa_oracle_mask_to_index(const uint8_t *mask, int64_t n_rows, int nKB, int32_t *row_ptr,
                                 int32_t *col_idx, uint32_t *bitmap)
{
    if (!mask || n_rows <= 0 || nKB <= 0) return -1;
    const int W = (nKB + 31) / 32;
    int64_t nnz = 0;
    for (int64_t r = 0; r < n_rows; ++r) {
        if (row_ptr) row_ptr[r] = (int32_t)nnz;
        for (int w = 0; w < W; ++w)
            if (bitmap) bitmap[r * W + w] = 0u;
        for (int j = 0; j < nKB; ++j)
            if (mask[r * nKB + j]) {
                if (col_idx) col_idx[nnz] = j;
                if (bitmap) bitmap[r * W + j / 32] |= (1u << (j % 32));
                ++nnz;
            }
    }
    if (row_ptr) row_ptr[n_rows] = (int32_t)nnz;
    return nnz;
}

/* ---------------------------------------------------------------------- */
/* [P1] §4.1 + §4.3 block-sparse attention written as its definition      */
/* (reading R4, R5): every key of the row is scored, keys in blocks the    */
/* mask switches off get -inf, then a two-pass softmax.                    */
/* Q, K, V: [n_heads][N][d] fp32; mask: [n_heads][nQB][nKB];               */
/* rows: global row ids (head * N + r) to evaluate; O: [n_rows][d];        */
/* LSE: [n_rows] (natural log).                                            */
int bsa_oracle_attention(const float *Q, const float *K, const float *V, int64_t n_heads,
                         int64_t N, int d, int bs, const uint8_t *mask, double scale,
                         const int64_t *rows, int64_t n_rows, double *O, double *LSE)
{
    if (!Q || !K || !V || !mask || !rows || !O || !LSE || n_heads <= 0 || N <= 0 || d <= 0 ||
        bs <= 0 || n_rows < 0)
        return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < n_rows; ++t)
        if (rows[t] < 0 || rows[t] >= n_heads * N) return ORACLE_ERR_ARG;
    /* reading R20: a ragged last block holds the keys up to N; nothing past N exists */
    const int64_t nB = (N + bs - 1) / bs;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        if (!s) {
#pragma omp atomic write
            err = ORACLE_ERR_ARG;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < n_rows; ++t) {
            if (!s) continue;
            const int64_t h = rows[t] / N, r = rows[t] % N, i = r / bs;
            const float *q = Q + (h * N + r) * d;
            /* scores over the whole row; inactive blocks get -inf */
            for (int64_t c = 0; c < N; ++c) {
                if (mask[(h * nB + i) * nB + c / bs]) {
                    const float *k = K + (h * N + c) * d;
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e) dot += (double)q[e] * (double)k[e];
                    s[c] = scale * dot;
                } else {
                    s[c] = -INFINITY;
                }
            }
            /* pass 1: row maximum */
            double m = -INFINITY;
            for (int64_t c = 0; c < N; ++c)
                if (s[c] > m) m = s[c];
            double *o = O + t * d;
            for (int e = 0; e < d; ++e) o[e] = 0.0;
            if (m == -INFINITY) { /* R5: no active key */
                LSE[t] = -INFINITY;
                continue;
            }
            /* pass 2: normaliser and weighted sum of values */
            double l = 0.0;
            for (int64_t c = 0; c < N; ++c) {
                double p = exp(s[c] - m); /* exp(-inf) = 0 for skipped keys */
                if (p == 0.0) continue;
                l += p;
                const float *v = V + (h * N + c) * d;
                for (int e = 0; e < d; ++e) o[e] += p * (double)v[e];
            }
            for (int e = 0; e < d; ++e) o[e] /= l;
            LSE[t] = m + log(l);
        }
        free(s);
    }
    return err;
}
