/*
 * kara.h -- C ABI of the GB300 (sm_103a) library for Kara's decode-time
 * KV-cache compression step.
 *
 * The method comes from "Kara: Sliding-Window KV Cache Compression for
 * Efficient Serving of Reasoning LLMs under Memory Constraints" (arXiv
 * 2607.01237; abstract and Section 1) and the gist.science technical summary
 * of that paper (sections "1. Sliding-Window Bidirectional Attention
 * Scoring", "2. Token2Chunk Module", "3. KvLLM Framework and Periodic
 * Compression").  For every window u = (sequence s, layer l, KV head g) the
 * step scores the W most recent tokens' keys with the queries of all W window
 * tokens, picks Top-K candidates, expands them into chunks under a retention
 * budget and packs the retained K/V rows into fresh paged blocks.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless their name starts with h_.
 *   - The caller owns all memory.  No entry point allocates device memory and
 *     none synchronises the stream, except kara_get_error, which waits for it.
 *   - Calls are asynchronous on `stream`.  The return value is the result of
 *     the host-side argument checks only; KARA_OK means the work was enqueued.
 *   - Device-side failures (a length shorter than the window, a block id
 *     outside the pool, a fresh list that is too short) are recorded in the
 *     caller's device word `err` (int32): the first error code wins, later
 *     ones are dropped.  The caller zeroes `err` before a step;
 *     kara_compress_batch zeroes it itself.  Read it with kara_get_error.
 *   - bf16 everywhere for Q, K and V; rows of head_dim elements are
 *     contiguous and 16-byte aligned.
 *
 * Notation: L cached length, W window, ws = L - W, B protected buffer,
 * C = W - B compressible keys, G = num_q_heads / num_kv_heads (query heads
 * g*G .. g*G+G-1 belong to KV head g), D head dim, bs block size,
 * p0 = floor(ws / bs), L' = L - C + R.
 *
 * Supported shapes: D in {64, 128}; block_size 16; 1 <= G <= 8;
 * W a multiple of 64 with 64 <= W <= 2048 and G*W <= 8192;
 * 1 <= K <= min(C, 1024); 1 <= R <= C.  Anything else returns
 * KARA_EUNSUPPORTED or KARA_EINVAL.
 */
#ifndef KARA_H
#define KARA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *kara_stream_t;

typedef enum {
    KARA_OK = 0,
    KARA_EINVAL = -1,        /* an argument or a cached length is out of range */
    KARA_EUNSUPPORTED = -2,  /* a shape outside the supported set above */
    KARA_ENOBLOCKS = -3,     /* the fresh-block list is shorter than the plan needs */
    KARA_EDUPBLOCK = -4,     /* a fresh block id repeats, or is a block the batch still lists (device) */
    KARA_ECUDA = -5,         /* a CUDA runtime call failed (launch or attribute) */
    KARA_EBADBLOCK = -6,     /* a block id outside [0, num_blocks) (device) */
    KARA_ETIMEOUT = -7,      /* a bounded device-side wait ran out (device) */
    KARA_EWORKSPACE = -8     /* workspace missing or smaller than kara_workspace_size */
} kara_status;

/*
 * Scoring and selection variants.  Mode 0 of each is the method as the pages
 * describe it.  The others are the ablations the summary's "Experimental
 * Results" (ablation studies) reports -- scores without bidirectional
 * attention, selection without Token2Chunk -- and the fixed-size chunks with
 * rigid boundaries its "Problem Statement" (item 2) sets Token2Chunk against.
 */
typedef enum {
    KARA_SCORE_BIDIRECTIONAL = 0,  /* every window query attends to all W window keys */
    KARA_SCORE_CAUSAL = 1          /* window query i attends to window keys j <= i only */
} kara_score_mode;

typedef enum {
    KARA_SELECT_TOKEN2CHUNK = 0,   /* Top-K candidates expanded into chunks (kara_select) */
    KARA_SELECT_TOP_R = 1,         /* the R positions first in score order, no chunks */
    KARA_SELECT_FIXED_CHUNK = 2    /* chunks [k*chunk, (k+1)*chunk) ranked by mean score */
} kara_select_mode;

/* Method parameters.  R is an explicit token count per window.  A zeroed
 * score_mode / select_mode / chunk gives the method as described. */
typedef struct {
    int32_t W;       /* window: the W most recent tokens of a sequence */
    int32_t B;       /* protected buffer at the end of the window, 0 <= B < W */
    int32_t K;       /* Top-K candidates per window */
    int32_t R;       /* tokens each window keeps out of its C compressible ones */
    float lambda;    /* chunk length penalty in (s_a + s_b) / (1 + lambda * len) */
    int32_t score_mode;   /* kara_score_mode */
    int32_t select_mode;  /* kara_select_mode */
    int32_t chunk;        /* chunk length for KARA_SELECT_FIXED_CHUNK, 1 <= chunk <= C; else ignored */
} kara_params;

/* Paged K/V pools.  Element (l, blk, g, slot, d) of a pool lives at
 *   base + l*layer_stride + blk*block_stride + g*head_stride + slot*head_dim + d
 * (strides in elements).  The canonical layout is
 * [num_layers][num_blocks][num_kv_heads][block_size][head_dim]. */
typedef struct {
    void *k;
    void *v;
    int64_t layer_stride, block_stride, head_stride;
    int32_t num_layers, num_blocks, num_kv_heads, num_q_heads, head_dim, block_size;
} kara_cache;

/* The sequences compressed by one call. */
typedef struct {
    int32_t n;                /* number of sequences */
    const int32_t *len;       /* device [n]: cached length L of each sequence */
    int32_t *block_table;     /* device [n][bt_stride]: logical block -> physical id */
    int32_t bt_stride;
    const void *q;            /* device bf16 [n][num_layers][num_q_heads][W][head_dim]:
                                 query states of each sequence's W window tokens */
} kara_batch;

/* Human-readable name of a status code (static storage). */
const char *kara_status_string(int status);

/* ABI version of this library. */
int kara_version(void);

/*
 * Host-only page plan (summary section 3, "Periodic Compression Policy": the
 * trailing blocks of selected sequences are compressed and memory is freed).
 * For each sequence: n_old = ceil(L/bs) - p0 blocks are released and
 * n_new = ceil(L'/bs) - p0 fresh blocks are taken.  Lets a caller size the
 * fresh and freed lists before kara_compact / kara_compress_batch.
 * h_len [n] host; h_n_new, h_n_old [n] host outputs (may be NULL);
 * h_total_new, h_total_old: sums (may be NULL).
 * Returns KARA_EINVAL if a length is below W or needs more than bt_stride blocks.
 */
kara_status kara_plan(const kara_params *p, int32_t block_size, int32_t n, const int32_t *h_len,
                      int32_t bt_stride, int32_t *h_n_new, int32_t *h_n_old,
                      int64_t *h_total_new, int64_t *h_total_old);

/* Bytes of device workspace kara_compact and kara_compress_batch need for n
 * sequences (256-byte aligned pieces; pass at least this many). */
size_t kara_workspace_size(const kara_cache *c, const kara_params *p, int32_t n);

/*
 * Window scores (summary section 1, "Mechanism"/"Rationale"; abstract:
 * bidirectional attention scores and selects KV pairs).  For every window,
 * every query head h of the group and every window query i < W:
 *     p[h,i,j] = softmax_j( <q_{h,i}, k_j> / sqrt(D) ),  j < W  (no causal mask)
 * and  scores[u][j] = sum_h sum_i p[h,i,j]  for the compressible keys j < C.
 * With score_mode KARA_SCORE_CAUSAL (an ablation) the softmax of query i runs
 * over the keys j <= i only and p[h,i,j] = 0 for j > i.
 * k_j is the key at logical position ws + j, read through the block table.
 * Logits accumulate in fp32 from bf16; the softmax and sums are fp32.
 * scores: device float [n][num_layers][num_kv_heads][C].
 * ws/ws_bytes: device workspace; kara_workspace_size bytes always suffice.
 * err: device int32 (see conventions); a window with a bad block id or a
 * length below W records the error and writes zeros.
 */
kara_status kara_score(const kara_cache *c, const kara_params *p, const kara_batch *b,
                       float *scores, void *ws, size_t ws_bytes, int32_t *err,
                       kara_stream_t stream);

/*
 * The window-query ring (the pages do not say where window queries live;
 * summary section 1 "Mechanism": the queries of all W window tokens score the
 * window).  b->q may hold, per (sequence, layer, query head), the queries of
 * the last W positions in a ring of W rows, the query of logical position x in
 * row x mod W.  Bidirectional scores do not depend on the order of the query
 * rows, so kara_score and kara_compress_batch read the ring as it stands
 * (score_mode KARA_SCORE_BIDIRECTIONAL; the causal ablation needs the rows in
 * position order).
 *
 * kara_compact_queries: after kara_compact / kara_compress_batch, moves the
 * queries of the kept rows and of the protected buffer to their new positions,
 * in place:  row (ws + r) mod W <- row (ws + kept[r]) mod W for r < R, and
 * row (ws + R + b) mod W <- row (L - B + b) mod W for b < B, where L is the
 * length before the step (b->len, as passed to the step) and kept is the
 * step's output.  Other rows are left as they are (positions past L', which
 * decoding overwrites).  Nothing moves if *err is non-zero (the step failed);
 * a kept row that is not strictly increasing in [0, C) records KARA_EINVAL and
 * leaves that window's queries as they are.  The next compression of a
 * sequence sees the queries of its whole window only if at least C - R tokens
 * were decoded since the last one (earlier positions' queries have left the
 * ring).
 *
 * kara_append_queries: one decode step; q_new [n][num_layers][num_q_heads][D]
 * (bf16, device) goes to row len[s] mod W of each ring, len[s] being the new
 * token's position (the length before the append).
 */
kara_status kara_compact_queries(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                 const int32_t *kept, int32_t *err, kara_stream_t stream);
kara_status kara_append_queries(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                const void *q_new, kara_stream_t stream);

/*
 * Decode attention over the paged cache (summary section 3: Kara adapted to
 * PagedAttention; the blocks a compression frees serve more decoding
 * sequences).  It reads K and V through the same block table that
 * kara_compact rewrites, so it is the consumer of the step's output.  For
 * each of n sequences and each query head h (KV head g = h / G):
 *     out[s][h] = sum_{x < len[s]} softmax_x(<q[s][h], k_x> / sqrt(D)) v_x
 * over the keys of layer `layer`, k_x and v_x at logical position x read
 * through block_table.  Logits are sums of exact bf16 products in fp32; the
 * softmax is fp32; each fp32 weight enters the weighted sum of V as two bf16
 * terms (relative error about 2^-17) with fp32 accumulation; fp32 output.
 * len [n] (device); block_table [n][bt_stride] (device); q: bf16
 * [n][num_q_heads][head_dim] (device, 16-byte aligned); out: float
 * [n][num_q_heads][head_dim] (device).
 * ws/ws_bytes: at least kara_decode_workspace_size(c, n, bt_stride) bytes.
 * err: device int32; a length outside [1, bt_stride*block_size] records
 * KARA_EINVAL and that sequence's output is 0; a block id outside the pool
 * records KARA_EBADBLOCK (the row is read as zeros, never from outside the pool);
 * K/V slices are staged through shared memory behind bounded waits, and one
 * that runs out records KARA_ETIMEOUT (outputs are then unspecified).
 * Returns KARA_ECUDA, before any launch, if the TMA tensor map over a pool
 * cannot be encoded (a stride of 2^40 bytes or more, for one).
 * Two launches on `stream`, both programmatic dependents of what precedes
 * them (the splits wait for the stream's previous kernel to complete before
 * reading anything; the merge waits for the splits); the call may be captured
 * into a CUDA graph.
 * Layout: each (block, KV head) slice of a pool must be block_size * head_dim
 * contiguous bf16 (rows at stride head_dim), as in the layout above.
 * Supported: the kara_cache shapes above; n <= 65535; bt_stride * block_size up to
 * 65535 * 1024 keys (the key splits of a sequence).
 */
size_t kara_decode_workspace_size(const kara_cache *c, int32_t n, int32_t bt_stride);
kara_status kara_decode_attention(const kara_cache *c, int32_t layer, int32_t n, const int32_t *len,
                                  const int32_t *block_table, int32_t bt_stride, const void *q, float *out,
                                  void *ws, size_t ws_bytes, int32_t *err, kara_stream_t stream);

/*
 * Top-K and Token2Chunk (summary section 1 "Selection"; section 2 "Process").
 * (select_mode KARA_SELECT_TOP_R and KARA_SELECT_FIXED_CHUNK replace the
 * chunk step, keeping cand as below: kept is the R first positions in the
 * score order; or chunks [k*chunk, min(C,(k+1)*chunk)) scored by their mean
 * -- a float sum in index order divided by the length -- visited by (mean
 * desc, start asc), kept whole when they fit R, then filled to exactly R with
 * other positions in score order.)
 * For each of n_windows windows with C fp32 scores:
 *   cand: the K positions first in the order (score desc, index asc), sorted
 *         by index.
 *   chunks: [c_t, c_{t+1}] for t < K-1, scored
 *         (s[a] + s[b]) / fmaf(lambda, len, 1), len = b - a + 1, in fp32 with
 *         round-to-nearest and no contraction; visited by (score desc, a asc)
 *         and kept when the tokens they add fit R (first fit); then the
 *         budget is filled to exactly R with candidates, then with other
 *         positions, both in score order.
 *   kept: the R retained positions, ascending.
 * scores [n_windows][C], cand [n_windows][K] (may be NULL), kept [n_windows][R].
 * The order is the one stated for finite scores (-0.0 counts as +0.0); NaN
 * scores still give a deterministic selection and never an out-of-range access.
 */
kara_status kara_select(const kara_params *p, int64_t n_windows, const float *scores,
                        int32_t *cand, int32_t *kept, kara_stream_t stream);

/*
 * Gather-compaction and block-table rewrite (summary section 3: Kara adapted
 * to PagedAttention).  For every sequence, layer, KV head and each of K and V,
 * the new logical positions from p0*bs on are filled with
 *     [p0*bs, ws)  <- the same old positions (head of the partial block),
 *     ws + r       <- old ws + kept[u][r], r < R,
 *     ws + R + b   <- old L - B + b, b < B (protected buffer, verbatim),
 * written into fresh blocks taken in sequence order from `fresh`.  Only fresh
 * blocks are written; old blocks are only read.  Then, if *err is still 0, the
 * table entries [p0, p0 + n_new) become the fresh ids, entries
 * [p0 + n_new, ceil(L/bs)) become -1, the released ids go to `freed` (in
 * sequence order) and new_len[s] = L'.  If *err is non-zero nothing is
 * committed: the table is unchanged, freed is untouched, new_len[s] = L.
 * Before anything is written the device checks (the pages give no rule: these
 * follow from filling caller-supplied blocks while the old ones are still
 * read) and records, with this precedence:
 *   KARA_EDUPBLOCK  a fresh id the plan consumes (fresh[i], i < total_new)
 *                   equals an earlier consumed id or an entry below
 *                   ceil(L/bs) of any table of the batch (values compared as
 *                   given; ids past total_new are never read);
 *   KARA_EBADBLOCK  a consumed fresh id outside [0, num_blocks);
 *   KARA_EINVAL     a kept row that is not strictly increasing in [0, C).
 * With any of these (or a plan error) no block is written.  An old block id
 * outside the pool, met while copying, records KARA_EBADBLOCK: fresh blocks
 * may then have been written, live blocks never are.
 * kept [n][num_layers][num_kv_heads][R]; fresh [n_fresh] (at least the plan's
 * total_new); freed [total_old]; new_len [n].
 * ws/ws_bytes: workspace of kara_workspace_size bytes.
 */
kara_status kara_compact(const kara_cache *c, const kara_params *p, const kara_batch *b,
                         const int32_t *kept, const int32_t *fresh, int64_t n_fresh,
                         int32_t *freed, int32_t *new_len, int32_t *err,
                         void *ws, size_t ws_bytes, kara_stream_t stream);

/*
 * The whole step for a batch: zero *err, plan, score, select, compact and
 * commit, without a host synchronisation: the work is ordered after what
 * `stream` already holds, and what is queued on `stream` afterwards runs after
 * all of it.  scores_out, cand_out, kept_out may be NULL (then the workspace
 * holds them); when given they receive [n][layers][Hkv][C], [..][K], [..][R].
 * Large batches are pipelined (kara_batch_groups): the sequences are split into
 * groups, and the selection and compaction of one group run on a second,
 * lower-priority stream while the next group is scored on a higher-priority
 * one; both streams are created for the call, forked from and joined back to
 * `stream`, and released when the call returns (CUDA frees them once their
 * work completes).  The fresh-id check covers the whole batch before any block
 * is written, and the tables are committed for the whole batch after every
 * copy, only if no error was recorded; a scoring error met in a later group
 * leaves fresh blocks of earlier groups written, never a live block.  A
 * stream that is being captured into a graph gets the unpipelined sequence.
 * phase_events: NULL, or 5 cudaEvent_t handles (cast to void *) recorded at
 * the start, after the plan, after scoring (the last group's), after
 * selection (pipelined: once the selection and compaction of every group have
 * joined `stream`) and after compaction + commit (pipelined: the commit), for
 * callers that time the phases.
 */
kara_status kara_compress_batch(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                const int32_t *fresh, int64_t n_fresh, int32_t *freed,
                                int32_t *new_len, float *scores_out, int32_t *cand_out,
                                int32_t *kept_out, void *ws, size_t ws_bytes, int32_t *err,
                                kara_stream_t stream, void *const *phase_events);

/*
 * Number of sequence groups kara_compress_batch pipelines this batch into (1:
 * scoring, selection and compaction run one after another), or a negative
 * status when the arguments are invalid.  Groups are used when the scoring
 * kernel leaves at least 4 SMs of the current device idle and each of its
 * resident clusters scores at least 32 windows per group; at most 8 groups,
 * at most one per sequence.  The environment variable KARA_BATCH_GROUPS=<m>
 * overrides the choice (clamped to [1, min(n, 64)]).
 */
int32_t kara_batch_groups(const kara_cache *c, const kara_params *p, const kara_batch *b);

/* Waits for `stream`, reads *err and returns it as a status (KARA_ECUDA if the
 * copy itself fails). */
kara_status kara_get_error(const int32_t *err, kara_stream_t stream);

/* Most sequences one kara_compact_static call accepts. */
#define KARA_STATIC_MAX_SEQS 8192

/*
 * kara_compact_static -- kara_compact without a workspace.  The paper has no
 * counterpart; this is a deployment convenience.
 *
 * For callers that cannot get device memory when compaction runs: a serving
 * engine whose memory pool handed all free HBM to the KV cache at start-up,
 * or a host program that embeds this library without any device allocator.
 * Such a caller passes its inputs and outputs exactly as for kara_compact
 * (same meaning, layout, ownership, checks and commit rule) but no workspace; the
 * per-sequence plan lives in a fixed array inside the library instead:
 * KARA_STATIC_MAX_SEQS entries of 32 bytes (256 KiB), held by every GPU that
 * loads the library until the process exits.
 *   - More than KARA_STATIC_MAX_SEQS sequences: returns KARA_EUNSUPPORTED
 *     before any device work.  Split the batch.
 *   - Each call looks up the array's device address in the current context
 *     (a host-side query that allocates nothing), so no address is kept past
 *     the context it belongs to (for example across cudaDeviceReset).
 *   - Every call uses the same array and it keeps the last call's contents.
 *     Nothing has to be cleared between calls (each call writes every entry
 *     it reads), but calls whose work overlaps on the GPU -- two streams with
 *     no ordering between them, or two host threads -- race on the array and
 *     corrupt each other's plan.  Calls ordered on one stream are safe.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *     routine.
 */
kara_status kara_compact_static(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                const int32_t *kept, const int32_t *fresh, int64_t n_fresh,
                                int32_t *freed, int32_t *new_len, int32_t *err,
                                kara_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KARA_H */
