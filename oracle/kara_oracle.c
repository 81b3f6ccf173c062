/*
 * kara_oracle.c -- plain, slow CPU oracle for Kara's decode-time KV-cache
 * compression step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the reference that the CUDA library
 * is checked against.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load it; the library never does.  It
 * shares no code, header, table or constant with the CUDA sources.
 *
 * Source of the method: "Kara: Sliding-Window KV Cache Compression for
 * Efficient Serving of Reasoning LLMs under Memory Constraints" (arXiv
 * 2607.01237) -- its abstract and Section 1 -- and the gist.science technical
 * summary of that paper, sections "1. Sliding-Window Bidirectional Attention
 * Scoring", "2. Token2Chunk Module" and "3. KvLLM Framework and Periodic
 * Compression"; the ablation variants (causal scores, token-level Top-R,
 * fixed-size chunks) follow its "Experimental Results" (ablation studies) and
 * "Problem Statement" (item 2); decode attention over the compacted cache
 * follows section "3. KvLLM Framework and Periodic Compression".  The pages
 * give no formula; every reading taken where they are silent is named at the
 * function that takes it.
 *
 * Notation, per window u = (sequence s, layer l, KV head g):
 *   L  cached length, W window, ws = L - W window start (logical position),
 *   B  protected buffer, C = W - B compressible keys,
 *   G  query heads per KV head (heads g*G .. g*G+G-1), D head dim,
 *   sigma = 1/sqrt(D), K Top-K, R retained tokens, lambda chunk penalty,
 *   bs block size, p0 = floor(ws/bs), o = ws mod bs.
 *
 * Precision: bf16 inputs are widened exactly to double; logits, softmax and
 * score sums are computed in double and each score is rounded once to float.
 * Selection works on float scores with float arithmetic in a fixed order
 * (build with -ffp-contract=off).  Compaction copies bytes.
 *
 * Parity pins: every function here is pinned by the not-GPU tests against
 * invariants, closed forms, brute force and an independent library softmax;
 * the chunk-score formula, lambda, the softmax scope and the budget rounding
 * are readings of silent passages and are pinned only to those readings.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t n_seq, layers, hq, hkv, d, block;
    int32_t W, B, K, R;
    float lambda;
    int32_t bt_stride, num_blocks;
    int64_t layer_stride, block_stride, head_stride; /* in elements; rows are d contiguous */
} kro_shape;

enum { KRO_OK = 0, KRO_EINVAL = -1, KRO_ENOBLOCKS = -3, KRO_EDUPBLOCK = -4, KRO_EBADBLOCK = -6 };

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int kro_version(void) { return 1; }

int kro_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Physical row of logical position x of sequence s in a pool, or NULL when the
 * block id is outside the pool. */
static const uint16_t *pool_row(const kro_shape *sh, const uint16_t *pool, const int32_t *bt,
                                int s, int l, int g, int64_t x)
{
    int32_t blk = bt[(int64_t)s * sh->bt_stride + x / sh->block];
    if (blk < 0 || blk >= sh->num_blocks) return NULL;
    return pool + (int64_t)l * sh->layer_stride + (int64_t)blk * sh->block_stride
                + (int64_t)g * sh->head_stride + (x % sh->block) * (int64_t)sh->d;
}

/*
 * Window scores (summary section 1, "Mechanism" and "Rationale"; the
 * abstract: KV pairs are scored and selected with bidirectional attention).
 *
 * The query states of ALL W window tokens score the keys of the window with no
 * causal mask.  For each query head h of the group and each window query i:
 *     l[j] = sigma * <q_{h,i}, k_j>,  j in [0, W)
 *     p[j] = exp(l[j] - max l) / sum_{j' < W} exp(l[j'] - max l)
 * and the weights are accumulated:  t[j] = sum_h sum_i p[j].
 * The score of compressible key j < C is s[j] = t[j] rounded to float.
 *
 * Readings where the pages are silent: sigma = 1/sqrt(D); the softmax runs
 * over all W window keys (buffer keys included, so sum_{j<W} t[j] = G*W and
 * sum_{j<C} s[j] <= G*W); heads of a GQA group are summed; no pooling.
 * k_j is the key at logical position ws + j, found through the block table.
 *
 * q: bf16 bits [n_seq][layers][hq][W][d]; kpool: bf16 bits, strides in sh;
 * scores: [n_seq][layers][hkv][C]; colsum (optional): [n_seq][layers][hkv][W].
 */
static int scores_impl(const kro_shape *sh, int causal, const uint16_t *q, const uint16_t *kpool,
                       const int32_t *bt, const int32_t *len, float *scores, double *colsum, int nthreads)
{
    const int W = sh->W, C = sh->W - sh->B, D = sh->d;
    const int G = sh->hq / sh->hkv;
    const int64_t nwin = (int64_t)sh->n_seq * sh->layers * sh->hkv;
    const double sigma = 1.0 / sqrt((double)D);
    int status = KRO_OK;
    if (W < 1 || C < 1 || sh->hq % sh->hkv != 0) return KRO_EINVAL;
    for (int s = 0; s < sh->n_seq; ++s)
        if (len[s] < W || (len[s] + sh->block - 1) / sh->block > sh->bt_stride) return KRO_EINVAL;
    if (nthreads < 1) nthreads = 1;

#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t u = 0; u < nwin; ++u) {
        const int s = (int)(u / ((int64_t)sh->layers * sh->hkv));
        const int l = (int)((u / sh->hkv) % sh->layers);
        const int g = (int)(u % sh->hkv);
        const int64_t ws = (int64_t)len[s] - W;
        double *kd = (double *)malloc(sizeof(double) * (size_t)W * D);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *lg = (double *)malloc(sizeof(double) * (size_t)W);
        double *t = (double *)calloc((size_t)W, sizeof(double));
        int bad = 0;
        for (int j = 0; j < W && !bad; ++j) {
            const uint16_t *row = pool_row(sh, kpool, bt, s, l, g, ws + j);
            if (!row) { bad = 1; break; }
            for (int e = 0; e < D; ++e) kd[(size_t)j * D + e] = bf16_to_double(row[e]);
        }
        if (!bad) {
            for (int r = 0; r < G; ++r) {
                const int h = g * G + r;
                for (int i = 0; i < W; ++i) {
                    const uint16_t *qrow = q + ((((int64_t)s * sh->layers + l) * sh->hq + h) * W + i) * D;
                    for (int e = 0; e < D; ++e) qd[e] = bf16_to_double(qrow[e]);
                    const int nk = causal ? i + 1 : W;  /* keys this query attends to */
                    double m = -INFINITY;
                    for (int j = 0; j < nk; ++j) {
                        double acc = 0.0;
                        for (int e = 0; e < D; ++e) acc += qd[e] * kd[(size_t)j * D + e];
                        lg[j] = sigma * acc;
                        if (lg[j] > m) m = lg[j];
                    }
                    double Z = 0.0;
                    for (int j = 0; j < nk; ++j) Z += exp(lg[j] - m);
                    for (int j = 0; j < nk; ++j) t[j] += exp(lg[j] - m) / Z;
                }
            }
            for (int j = 0; j < C; ++j) scores[u * C + j] = (float)t[j];
            if (colsum)
                for (int j = 0; j < W; ++j) colsum[u * W + j] = t[j];
        } else {
#pragma omp atomic write
            status = KRO_EBADBLOCK;
        }
        free(kd); free(qd); free(lg); free(t);
    }
    return status;
}

int kro_scores(const kro_shape *sh, const uint16_t *q, const uint16_t *kpool, const int32_t *bt,
               const int32_t *len, float *scores, double *colsum, int nthreads)
{
    return scores_impl(sh, 0, q, kpool, bt, len, scores, colsum, nthreads);
}

/*
 * Causal window scores: the ablation that removes bidirectional scoring
 * (summary, "Experimental Results", ablation studies: removing the
 * bidirectional attention scoring costs accuracy).  Reading: without it, each
 * window query attends as in decoding, to the window keys at or before its own
 * position only:
 *     p[j] = exp(l[j] - max) / sum_{j' <= i} exp(l[j'] - max)  for j <= i,
 *     p[j] = 0                                                 for j >  i,
 * with max over j <= i; everything else is as in kro_scores (so still
 * sum_{j<W} t[j] = G*W).
 */
int kro_scores_causal(const kro_shape *sh, const uint16_t *q, const uint16_t *kpool, const int32_t *bt,
                      const int32_t *len, float *scores, double *colsum, int nthreads)
{
    return scores_impl(sh, 1, q, kpool, bt, len, scores, colsum, nthreads);
}

/*
 * Decode attention over the paged cache: the reader of the tables the step
 * rewrites (summary section 3, "KvLLM Framework and Periodic Compression":
 * Kara adapted to PagedAttention, and the freed memory serves more decoding
 * sequences).  One decode query per sequence and query head h (KV head
 * g = h / G) attends to every cached key x in [0, L) of one layer:
 *     l[x] = sigma * <q_h, k_x>,   o_h = sum_x exp(l[x] - max l) v_x / sum_x exp(l[x] - max l)
 * in double from the exact bf16 values, each output element rounded once to
 * float.  Reading: plain decode attention with no mask inside the cache (the
 * pages name PagedAttention and print no kernel); sigma = 1/sqrt(D) as above.
 * q: bf16 bits [n_seq][hq][d]; out: float [n_seq][hq][d].
 */
int kro_decode_attention(const kro_shape *sh, int layer, const uint16_t *q, const uint16_t *kpool,
                         const uint16_t *vpool, const int32_t *bt, const int32_t *len, float *out, int nthreads)
{
    const int D = sh->d, G = sh->hq / sh->hkv;
    const double sigma = 1.0 / sqrt((double)D);
    int status = KRO_OK;
    if (layer < 0 || layer >= sh->layers || sh->hq % sh->hkv != 0) return KRO_EINVAL;
    for (int s = 0; s < sh->n_seq; ++s)
        if (len[s] < 1 || (len[s] + sh->block - 1) / sh->block > sh->bt_stride) return KRO_EINVAL;
    if (nthreads < 1) nthreads = 1;

#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t sh_idx = 0; sh_idx < (int64_t)sh->n_seq * sh->hq; ++sh_idx) {
        const int s = (int)(sh_idx / sh->hq), h = (int)(sh_idx % sh->hq), g = h / G;
        const int64_t L = len[s];
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *lg = (double *)malloc(sizeof(double) * (size_t)L);
        double *acc = (double *)calloc((size_t)D, sizeof(double));
        const uint16_t *qrow = q + ((int64_t)s * sh->hq + h) * D;
        for (int e = 0; e < D; ++e) qd[e] = bf16_to_double(qrow[e]);
        int bad = 0;
        double m = -INFINITY;
        for (int64_t x = 0; x < L && !bad; ++x) {
            const uint16_t *kr = pool_row(sh, kpool, bt, s, layer, g, x);
            if (!kr) { bad = 1; break; }
            double dot = 0.0;
            for (int e = 0; e < D; ++e) dot += qd[e] * bf16_to_double(kr[e]);
            lg[x] = sigma * dot;
            if (lg[x] > m) m = lg[x];
        }
        double Z = 0.0;
        for (int64_t x = 0; x < L && !bad; ++x) {
            const uint16_t *vr = pool_row(sh, vpool, bt, s, layer, g, x);
            const double w = exp(lg[x] - m);
            Z += w;
            for (int e = 0; e < D; ++e) acc[e] += w * bf16_to_double(vr[e]);
        }
        if (bad) {
#pragma omp atomic write
            status = KRO_EBADBLOCK;
        } else {
            for (int e = 0; e < D; ++e) out[sh_idx * D + e] = (float)(acc[e] / Z);
        }
        free(qd); free(lg); free(acc);
    }
    return status;
}

/* ---- selection ---------------------------------------------------------- */

/* The total order used everywhere in selection: j precedes j' when its score is
 * larger, or equal with the lower index (ties to the lower index is a reading:
 * the pages do not say how ties break). */
static int precedes(const float *s, int32_t a, int32_t b)
{
    return s[a] > s[b] || (s[a] == s[b] && a < b);
}

/* Stable merge sort of idx[0..n) by a "comes first" predicate over (key, index). */
typedef int (*first_fn)(const void *ctx, int32_t a, int32_t b);

static void merge_sort(int32_t *idx, int32_t *tmp, int n, first_fn first, const void *ctx)
{
    if (n < 2) return;
    int h = n / 2;
    merge_sort(idx, tmp, h, first, ctx);
    merge_sort(idx + h, tmp, n - h, first, ctx);
    int i = 0, j = h, k = 0;
    while (i < h && j < n) tmp[k++] = first(ctx, idx[j], idx[i]) ? idx[j++] : idx[i++];
    while (i < h) tmp[k++] = idx[i++];
    while (j < n) tmp[k++] = idx[j++];
    memcpy(idx, tmp, sizeof(int32_t) * (size_t)n);
}

static int first_by_score(const void *ctx, int32_t a, int32_t b)
{
    return precedes((const float *)ctx, a, b);
}

static int first_ascending(const void *ctx, int32_t a, int32_t b)
{
    (void)ctx;
    return a < b;
}

typedef struct { const float *cs; const int32_t *a; } chunk_ctx;

static int first_chunk(const void *ctx, int32_t x, int32_t y)
{
    const chunk_ctx *c = (const chunk_ctx *)ctx;
    return c->cs[x] > c->cs[y] || (c->cs[x] == c->cs[y] && c->a[x] < c->a[y]);
}

/*
 * Top-K candidates and Token2Chunk for one window.
 *
 * Top-K (summary section 1, "Selection"): the K positions first under the
 * order above, reported sorted by index.
 *
 * Token2Chunk (summary section 2, "Process"; abstract: "expand a subset of
 * selected KV pairs into chunks"): with candidates c_0 < ... < c_{K-1}, every
 * consecutive pair (c_t, c_{t+1}) bounds chunk t = [c_t, c_{t+1}] of
 * len = c_{t+1} - c_t + 1 tokens.  A chunk is scored from its length and its
 * endpoint scores.  Reading (the pages print no formula):
 *     cs = (s[a] + s[b]) / (1 + lambda * len)
 * evaluated in float as num = s[a] + s[b]; den = fmaf(lambda, len, 1); num/den.
 * Chunks are visited by (cs descending, a ascending) and a chunk is kept when
 * the tokens it adds to the kept set still fit the budget R; otherwise it is
 * skipped and the next one is tried (first fit).  The budget is then filled to
 * exactly R: first with candidates not yet kept, in score order, then with any
 * other compressible position, in score order.  Exactly R tokens per window is
 * a reading too: every (layer, head) of a sequence then keeps the same count,
 * so one block table stays valid for all of them.
 *
 * Outputs: cand[K] ascending, kept[R] ascending; optionally chunk_score[K-1]
 * and chunk_taken[K-1] in chunk (index) order.
 */
int kro_select(int C, int K, int R, float lambda, const float *s, int32_t *cand, int32_t *kept,
               float *chunk_score, uint8_t *chunk_taken)
{
    if (C < 1 || K < 1 || K > C || R < 1 || R > C) return KRO_EINVAL;
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)C);
    int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)C);
    uint8_t *in = (uint8_t *)calloc((size_t)C, 1);
    const int nch = K - 1;
    float *cs = (float *)malloc(sizeof(float) * (size_t)(nch > 0 ? nch : 1));
    int32_t *ca = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nch > 0 ? nch : 1));
    int32_t *corder = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nch > 0 ? nch : 1));

    /* Top-K under the score order, then by index. */
    for (int j = 0; j < C; ++j) order[j] = j;
    merge_sort(order, tmp, C, first_by_score, s);
    for (int t = 0; t < K; ++t) cand[t] = order[t];
    merge_sort(cand, tmp, K, first_ascending, NULL);

    /* Chunks between consecutive candidates and their scores. */
    for (int t = 0; t < nch; ++t) {
        const int32_t a = cand[t], b = cand[t + 1];
        const float num = s[a] + s[b];
        const float den = fmaf(lambda, (float)(b - a + 1), 1.0f);
        cs[t] = num / den;
        ca[t] = a;
        corder[t] = t;
    }
    chunk_ctx cc = { cs, ca };
    if (nch > 0) merge_sort(corder, tmp, nch, first_chunk, &cc);

    /* Greedy first fit under the budget. */
    int count = 0;
    for (int r = 0; r < nch; ++r) {
        const int t = corder[r];
        const int32_t a = cand[t], b = cand[t + 1];
        int add = 0;
        for (int32_t x = a; x <= b; ++x) add += !in[x];
        if (count + add <= R) {
            for (int32_t x = a; x <= b; ++x) in[x] = 1;
            count += add;
            if (chunk_taken) chunk_taken[t] = 1;
        } else if (chunk_taken) {
            chunk_taken[t] = 0;
        }
    }
    /* Fill 1: candidates not kept yet, in score order (the first K of order). */
    for (int r = 0; r < K && count < R; ++r)
        if (!in[order[r]]) { in[order[r]] = 1; ++count; }
    /* Fill 2: any other compressible position, in score order. */
    for (int r = K; r < C && count < R; ++r)
        if (!in[order[r]]) { in[order[r]] = 1; ++count; }

    int w = 0;
    for (int j = 0; j < C; ++j)
        if (in[j]) kept[w++] = j;
    if (chunk_score)
        for (int t = 0; t < nch; ++t) chunk_score[t] = cs[t];

    free(order); free(tmp); free(in); free(cs); free(ca); free(corder);
    return w == R ? KRO_OK : KRO_EINVAL;
}

/*
 * The two selection ablations.  Both keep the Top-K candidates (cand) of
 * kro_select and replace Token2Chunk:
 *
 * mode 1, token-level Top-R -- the ablation that removes Token2Chunk (summary,
 *   "Experimental Results", ablation studies), leaving isolated KV pairs
 *   (summary, "Problem Statement", item 2): kept = the R positions first in
 *   the score order, sorted by index.
 *
 * mode 2, fixed-size chunks with rigid boundaries (summary, "Problem
 *   Statement", item 2, the granularity Token2Chunk replaces).  Readings: the
 *   compressible region is cut into chunks [k*chunk, min(C, (k+1)*chunk)); a
 *   chunk scores the mean of its scores, summed in float in index order and
 *   divided by its length (round to nearest); chunks are visited by (mean
 *   desc, start asc) and kept whole when they fit the budget (first fit); the
 *   budget is then filled to exactly R with any other position in score order,
 *   as kro_select does.
 *
 * mode 0 is kro_select.  chunk is used by mode 2 only (1 <= chunk <= C).
 */
int kro_select_mode(int mode, int chunk, int C, int K, int R, float lambda, const float *s, int32_t *cand,
                    int32_t *kept)
{
    if (mode == 0) return kro_select(C, K, R, lambda, s, cand, kept, NULL, NULL);
    if (mode < 0 || mode > 2 || C < 1 || K < 1 || K > C || R < 1 || R > C) return KRO_EINVAL;
    if (mode == 2 && (chunk < 1 || chunk > C)) return KRO_EINVAL;
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)C);
    int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)C);
    uint8_t *in = (uint8_t *)calloc((size_t)C, 1);
    for (int j = 0; j < C; ++j) order[j] = j;
    merge_sort(order, tmp, C, first_by_score, s);
    for (int t = 0; t < K; ++t) cand[t] = order[t];
    merge_sort(cand, tmp, K, first_ascending, NULL);

    int count = 0;
    if (mode == 2) {
        const int nch = (C + chunk - 1) / chunk;
        float *mean = (float *)malloc(sizeof(float) * (size_t)nch);
        int32_t *start = (int32_t *)malloc(sizeof(int32_t) * (size_t)nch);
        int32_t *corder = (int32_t *)malloc(sizeof(int32_t) * (size_t)nch);
        int32_t *ctmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)nch);
        for (int k = 0; k < nch; ++k) {
            const int a = k * chunk, b = (k + 1) * chunk < C ? (k + 1) * chunk : C;
            float sum = 0.0f;
            for (int j = a; j < b; ++j) sum += s[j];
            mean[k] = sum / (float)(b - a);
            start[k] = a;
            corder[k] = k;
        }
        chunk_ctx cc = { mean, start };
        merge_sort(corder, ctmp, nch, first_chunk, &cc);
        for (int r = 0; r < nch; ++r) {
            const int k = corder[r];
            const int a = k * chunk, b = (k + 1) * chunk < C ? (k + 1) * chunk : C;
            if (count + (b - a) <= R) {
                for (int j = a; j < b; ++j) in[j] = 1;
                count += b - a;
            }
        }
        free(mean); free(start); free(corder); free(ctmp);
    }
    for (int r = 0; r < C && count < R; ++r)
        if (!in[order[r]]) { in[order[r]] = 1; ++count; }
    int w = 0;
    for (int j = 0; j < C; ++j)
        if (in[j]) kept[w++] = j;
    free(order); free(tmp); free(in);
    return w == R ? KRO_OK : KRO_EINVAL;
}

/* kro_select_mode over nwin windows laid out back to back. */
int kro_select_mode_batch(int mode, int chunk, int64_t nwin, int C, int K, int R, float lambda,
                          const float *scores, int32_t *cand, int32_t *kept, int nthreads)
{
    int status = KRO_OK;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads)
    for (int64_t u = 0; u < nwin; ++u) {
        int st = kro_select_mode(mode, chunk, C, K, R, lambda, scores + u * C, cand + u * K, kept + u * R);
        if (st != KRO_OK) {
#pragma omp atomic write
            status = st;
        }
    }
    return status;
}

/* kro_select over nwin windows laid out back to back: scores [nwin][C],
 * cand [nwin][K], kept [nwin][R]. */
int kro_select_batch(int64_t nwin, int C, int K, int R, float lambda, const float *scores,
                     int32_t *cand, int32_t *kept, int nthreads)
{
    int status = KRO_OK;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads)
    for (int64_t u = 0; u < nwin; ++u) {
        int st = kro_select(C, K, R, lambda, scores + u * C, cand + u * K, kept + u * R, NULL, NULL);
        if (st != KRO_OK) {
#pragma omp atomic write
            status = st;
        }
    }
    return status;
}

/* ---- paged plan and compaction -------------------------------------------- */

/*
 * Page plan (summary section 3, "Periodic Compression Policy": the trailing
 * blocks of a sequence are compressed and memory is freed).  After the step
 * the window keeps R compressible tokens plus the B buffer tokens, so
 *     L' = ws + R + B = L - C + R,
 * blocks before p0 = floor(ws/bs) are untouched, the old tail blocks
 * [p0, ceil(L/bs)) are all released (n_old of them) and the rebuilt tail
 * [p0, ceil(L'/bs)) takes n_new fresh blocks.  Rebuilding into fresh blocks
 * (rather than in place) is a reading: the pages do not say how pages are
 * rewritten.
 */
int kro_plan(int n, const int32_t *len, int W, int B, int R, int bs, int bt_stride,
             int32_t *n_new, int32_t *n_old)
{
    if (W < 1 || B < 0 || B >= W || R < 1 || R > W - B || bs < 1) return KRO_EINVAL;
    for (int s = 0; s < n; ++s) {
        const int64_t L = len[s];
        if (L < W || (L + bs - 1) / bs > bt_stride) return KRO_EINVAL;
        const int64_t ws = L - W, p0 = ws / bs;
        const int64_t Lp = ws + R + B;
        n_old[s] = (int32_t)((L + bs - 1) / bs - p0);
        n_new[s] = (int32_t)((Lp + bs - 1) / bs - p0);
    }
    return KRO_OK;
}

/*
 * Compaction of the window-query ring (a reading: the pages are silent on
 * where window queries live; the gist.science summary, section 1 "Mechanism",
 * only has the queries of all W window tokens score the window).  Each
 * (sequence, layer, query head) keeps the queries of its last W positions in
 * a ring of W rows, the query of logical position x in row x mod W.  When the
 * step compacts K and V, the queries of the rows it keeps move with them, to
 * the same new positions (kept row r to ws + r, buffer row b to ws + R + b):
 *     ring[(ws + r) mod W]     <- old ring[(ws + kept[r]) mod W],  r < R
 *     ring[(ws + R + b) mod W] <- old ring[(L - B + b) mod W],     b < B
 * where kept is the window's (KV head g = h / G) retained set.  All other
 * rows are left as they are (they belong to positions past L', which decoding
 * overwrites).  Reading: the queries keep their stored values, as K does.
 * q: bf16 bits [n_seq][layers][hq][W][d], modified in place; len: lengths
 * before the step; kept: [n_seq][layers][hkv][R].
 */
int kro_compact_queries(const kro_shape *sh, uint16_t *q, const int32_t *len, const int32_t *kept)
{
    const int W = sh->W, B = sh->B, R = sh->R, D = sh->d, G = sh->hq / sh->hkv;
    if (W < 1 || B < 0 || B >= W || R < 1 || R > W - B || sh->hq % sh->hkv) return KRO_EINVAL;
    for (int s = 0; s < sh->n_seq; ++s)
        if (len[s] < W) return KRO_EINVAL;
    uint16_t *old = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)W * D);
    for (int s = 0; s < sh->n_seq; ++s) {
        const int64_t L = len[s], ws = L - W;
        for (int l = 0; l < sh->layers; ++l)
            for (int h = 0; h < sh->hq; ++h) {
                uint16_t *ring = q + (((int64_t)s * sh->layers + l) * sh->hq + h) * W * D;
                const int32_t *kp = kept + (((int64_t)s * sh->layers + l) * sh->hkv + h / G) * R;
                memcpy(old, ring, sizeof(uint16_t) * (size_t)W * D);
                for (int r = 0; r < R; ++r)
                    memcpy(ring + ((ws + r) % W) * D, old + ((ws + kp[r]) % W) * D, sizeof(uint16_t) * (size_t)D);
                for (int b = 0; b < B; ++b)
                    memcpy(ring + ((ws + R + b) % W) * D, old + ((L - B + b) % W) * D, sizeof(uint16_t) * (size_t)D);
            }
    }
    free(old);
    return KRO_OK;
}

/*
 * Gather-compaction and block-table rewrite (summary section 3: Kara adapted
 * to PagedAttention, so the retained K/V must land in paged blocks).
 *
 * Per sequence s, with fresh ids consumed in sequence order, for every layer,
 * KV head and each of the K and V pools, new logical positions are filled:
 *     x in [p0*bs, ws)      <- old x           (head of the partial first block)
 *     ws + r, r < R         <- old ws + kept[r] (retained tokens, in order)
 *     ws + R + b, b < B     <- old L - B + b    (protected buffer, verbatim)
 * Old rows are read through the old table; new rows are written to the fresh
 * blocks.  Then freed[] receives the old tail ids, the table entries
 * [p0, p0 + n_new) become the fresh ids, entries [p0 + n_new, ceil(L/bs)) are
 * cleared to -1, and new_len[s] = L'.  Slots past L' in the last fresh block
 * are not written.
 *
 * kept: [n_seq][layers][hkv][R]; kpool/vpool/bt are modified in place.
 *
 * Inputs that would make the rewrite unsound are rejected before anything is
 * written (the pages give no rule; these follow from rebuilding into blocks
 * the caller supplies while the old ones are still read):
 *   - a fresh id consumed by the plan that repeats an earlier one, or that is
 *     an entry below ceil(L/bs) of any table of the batch (a block the batch
 *     still keeps or reads): KRO_EDUPBLOCK;
 *   - a fresh id outside the pool: KRO_EBADBLOCK;
 *   - a kept row that is not strictly increasing in [0, C): KRO_EINVAL
 *     (Top-K and Token2Chunk produce ascending positions).
 */
int kro_compact(const kro_shape *sh, uint16_t *kpool, uint16_t *vpool, int32_t *bt,
                const int32_t *len, const int32_t *kept, const int32_t *fresh, int64_t n_fresh,
                int32_t *freed, int32_t *new_len)
{
    const int W = sh->W, B = sh->B, R = sh->R, C = W - B, bs = sh->block, D = sh->d;
    int32_t *nn = (int32_t *)malloc(sizeof(int32_t) * (size_t)(sh->n_seq > 0 ? sh->n_seq : 1));
    int32_t *no = (int32_t *)malloc(sizeof(int32_t) * (size_t)(sh->n_seq > 0 ? sh->n_seq : 1));
    int st = kro_plan(sh->n_seq, len, W, B, R, bs, sh->bt_stride, nn, no);
    int64_t tot_new = 0;
    for (int s = 0; st == KRO_OK && s < sh->n_seq; ++s) tot_new += nn[s];
    if (st == KRO_OK && tot_new > n_fresh) st = KRO_ENOBLOCKS;
    /* every consumed fresh id against the earlier ones and against every live
       table entry of the batch, one pair at a time */
    for (int64_t i = 0; st == KRO_OK && i < tot_new; ++i) {
        for (int64_t j = 0; j < i; ++j)
            if (fresh[j] == fresh[i]) st = KRO_EDUPBLOCK;
        for (int s = 0; s < sh->n_seq; ++s) {
            const int64_t nb = ((int64_t)len[s] + bs - 1) / bs;
            for (int64_t lb = 0; lb < nb; ++lb)
                if (bt[(int64_t)s * sh->bt_stride + lb] == fresh[i]) st = KRO_EDUPBLOCK;
        }
    }
    for (int64_t i = 0; st == KRO_OK && i < tot_new; ++i)
        if (fresh[i] < 0 || fresh[i] >= sh->num_blocks) st = KRO_EBADBLOCK;
    const int64_t nwin = (int64_t)sh->n_seq * sh->layers * sh->hkv;
    for (int64_t w = 0; st == KRO_OK && w < nwin; ++w)
        for (int r = 0; r < R; ++r) {
            const int32_t k = kept[w * R + r];
            if (k < 0 || k >= C || (r > 0 && kept[w * R + r - 1] >= k)) st = KRO_EINVAL;
        }
    if (st != KRO_OK) { free(nn); free(no); return st; }

    int64_t off_new = 0, off_old = 0;
    for (int s = 0; s < sh->n_seq; ++s) {
        const int64_t L = len[s], ws = L - W, p0 = ws / bs;
        const int32_t *nbt = fresh + off_new;
        int32_t *row_bt = bt + (int64_t)s * sh->bt_stride;
        for (int64_t t = 0; t < no[s]; ++t) {
            int32_t b = row_bt[p0 + t];
            if (b < 0 || b >= sh->num_blocks) { free(nn); free(no); return KRO_EBADBLOCK; }
        }
        for (int l = 0; l < sh->layers; ++l)
            for (int g = 0; g < sh->hkv; ++g) {
                const int32_t *kp = kept + (((int64_t)s * sh->layers + l) * sh->hkv + g) * R;
                for (int which = 0; which < 2; ++which) {
                    uint16_t *pool = which ? vpool : kpool;
                    for (int64_t xn = p0 * bs; xn < ws + R + B; ++xn) {
                        int64_t xo;
                        if (xn < ws) xo = xn;
                        else if (xn < ws + R) xo = ws + kp[xn - ws];
                        else xo = L - B + (xn - ws - R);
                        const uint16_t *src = pool_row(sh, pool, bt, s, l, g, xo);
                        const int32_t blk = nbt[xn / bs - p0];
                        uint16_t *dst = pool + (int64_t)l * sh->layer_stride
                                        + (int64_t)blk * sh->block_stride
                                        + (int64_t)g * sh->head_stride + (xn % bs) * (int64_t)D;
                        memcpy(dst, src, sizeof(uint16_t) * (size_t)D);
                    }
                }
            }
        for (int64_t t = 0; t < no[s]; ++t) {
            freed[off_old + t] = row_bt[p0 + t];
            row_bt[p0 + t] = t < nn[s] ? nbt[t] : -1;
        }
        new_len[s] = (int32_t)(ws + R + B);
        off_new += nn[s];
        off_old += no[s];
    }
    free(nn); free(no);
    return KRO_OK;
}
