// Host side of the C ABI: argument checks, workspace layout and the launch
// sequence of each entry point.  No allocation, no stream synchronisation
// (except kara_get_error).
#include <stdlib.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include "kara_common.cuh"

using namespace kara;

namespace {

constexpr int kMaxK = 1024;
constexpr int kMaxG = 8;
constexpr int kMaxGW = 8192;  // query rows per window the scoring kernel keeps statistics for

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

kara_status check_params(const kara_params *p)
{
    if (!p) return KARA_EINVAL;
    if (p->W < 64 || p->W > 2048 || p->W % 64 != 0) return KARA_EUNSUPPORTED;
    if (p->B < 0 || p->B >= p->W) return KARA_EINVAL;
    const int C = p->W - p->B;
    if (p->K < 1 || p->K > C) return KARA_EINVAL;
    if (p->K > kMaxK) return KARA_EUNSUPPORTED;
    if (p->R < 1 || p->R > C) return KARA_EINVAL;
    if (!(p->lambda == p->lambda)) return KARA_EINVAL;  // NaN
    if (p->score_mode != KARA_SCORE_BIDIRECTIONAL && p->score_mode != KARA_SCORE_CAUSAL) return KARA_EINVAL;
    if (p->select_mode < KARA_SELECT_TOKEN2CHUNK || p->select_mode > KARA_SELECT_FIXED_CHUNK) return KARA_EINVAL;
    if (p->select_mode == KARA_SELECT_FIXED_CHUNK && (p->chunk < 1 || p->chunk > C)) return KARA_EINVAL;
    return KARA_OK;
}

kara_status check_cache(const kara_cache *c)
{
    if (!c || !c->k || !c->v) return KARA_EINVAL;
    if (c->head_dim != 64 && c->head_dim != 128) return KARA_EUNSUPPORTED;
    if (c->block_size != 16) return KARA_EUNSUPPORTED;
    if (c->num_kv_heads < 1 || c->num_q_heads < 1 || c->num_q_heads % c->num_kv_heads != 0)
        return KARA_EINVAL;
    if (c->num_q_heads / c->num_kv_heads > kMaxG) return KARA_EUNSUPPORTED;
    if (c->num_layers < 1 || c->num_blocks < 1) return KARA_EINVAL;
    if (!aligned16(c->k) || !aligned16(c->v)) return KARA_EINVAL;
    if (c->layer_stride % 8 || c->block_stride % 8 || c->head_stride % 8) return KARA_EINVAL;
    if (c->layer_stride < 0 || c->block_stride < 0 || c->head_stride < 0) return KARA_EINVAL;
    return KARA_OK;
}

kara_status make_geo(const kara_cache *c, const kara_params *p, const kara_batch *b, Geo *g)
{
    kara_status st = check_params(p);
    if (st != KARA_OK) return st;
    st = check_cache(c);
    if (st != KARA_OK) return st;
    if (!b || b->n < 0) return KARA_EINVAL;
    if (b->n > 0 && (!b->len || !b->block_table || !b->q || b->bt_stride < 1)) return KARA_EINVAL;
    if (b->q && !aligned16(b->q)) return KARA_EINVAL;
    if ((c->num_q_heads / c->num_kv_heads) * p->W > kMaxGW) return KARA_EUNSUPPORTED;
    memset(g, 0, sizeof *g);
    g->k = static_cast<const uint16_t *>(c->k);
    g->v = static_cast<const uint16_t *>(c->v);
    g->layer_stride = c->layer_stride;
    g->block_stride = c->block_stride;
    g->head_stride = c->head_stride;
    g->layers = c->num_layers;
    g->num_blocks = c->num_blocks;
    g->hkv = c->num_kv_heads;
    g->hq = c->num_q_heads;
    g->G = c->num_q_heads / c->num_kv_heads;
    g->D = c->head_dim;
    g->bs = c->block_size;
    g->W = p->W;
    g->B = p->B;
    g->C = p->W - p->B;
    g->K = p->K;
    g->R = p->R;
    g->lambda = p->lambda;
    g->n = b->n;
    g->bt_stride = b->bt_stride;
    g->len = b->len;
    g->bt = b->block_table;
    g->q = static_cast<const uint16_t *>(b->q);
    g->nwin = (int64_t)b->n * c->num_layers * c->num_kv_heads;
    g->causal = p->score_mode == KARA_SCORE_CAUSAL;
    return KARA_OK;
}

// Workspace layout of kara_compress_batch: [plan][scores][cand][kept][score scratch].
struct WsLayout {
    size_t plan, scores, cand, kept, scratch, total;
};

WsLayout layout(const Geo &g)
{
    WsLayout w;
    size_t off = 0;
    w.plan = off;
    off += align256((size_t)(g.n > 0 ? g.n : 1) * sizeof(SeqPlan));
    w.scores = off;
    off += align256((size_t)g.nwin * g.C * sizeof(float));
    w.cand = off;
    off += align256((size_t)g.nwin * g.K * sizeof(int32_t));
    w.kept = off;
    off += align256((size_t)g.nwin * g.R * sizeof(int32_t));
    w.scratch = off;
    off += score_scratch_bytes(g);
    w.total = off;
    return w;
}

template <class T>
T *at(void *ws, size_t off) { return reinterpret_cast<T *>(static_cast<char *>(ws) + off); }

kara_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KARA_OK : KARA_ECUDA; }

// ---- pipelined batches ------------------------------------------------------
// The single-pass scorer holds one CTA per SM on the SMs its resident clusters
// cover and leaves the rest idle (on GB300, 36 clusters of 4 CTAs take 144 of
// 152 SMs at W = 1024).  A large batch is therefore split into groups of
// sequences: the scoring of group i + 1 runs while the selection, kept-row check
// and copy of group i run on a second, lower-priority stream and take the idle
// SMs.  The fresh-id check of the whole batch runs before any copy and the table
// commit of the whole batch after every copy, so the call stays all-or-nothing
// for the tables; each group writes only its own sequences' fresh blocks.  The
// groups are scored one after another on one stream: while a group's last
// clusters finish, the queued selection and copy work also takes the SMs they
// leave (scoring the groups on two alternating streams measured slower, as that
// work then fell behind on the idle SMs alone).
constexpr int kMaxGroups = 8;
constexpr int kMinIdleSms = 4;           // fewer idle SMs: the overlap cannot pay for the groups' tails
constexpr int kWindowsPerCluster = 32;   // windows each resident cluster scores per group, at least

// Sequences [s0, s1) of a batch as a batch of their own.
Geo sub_batch(const Geo &g, int s0, int s1)
{
    Geo h = g;
    h.n = s1 - s0;
    h.len = g.len + s0;
    h.bt = g.bt + (int64_t)s0 * g.bt_stride;
    h.q = g.q + (int64_t)s0 * g.layers * g.hq * g.W * g.D;
    h.nwin = (int64_t)h.n * g.layers * g.hkv;
    return h;
}

// Groups of sequences kara_compress_batch splits batch g into (1: none).
// KARA_BATCH_GROUPS=<m> overrides the choice (clamped to [1, min(n, 64)]).
static_assert(kMaxGroups <= 64, "events of a pipelined call");
int batch_groups(const Geo &g)
{
    if (g.n < 2) return 1;
    if (const char *v = getenv("KARA_BATCH_GROUPS")) {
        const int m = atoi(v);
        const int cap = g.n < 64 ? g.n : 64;
        return m < 1 ? 1 : m > cap ? cap : m;
    }
    if (score_idle_sms(g) < kMinIdleSms) return 1;
    const int64_t nres = score_resident_clusters(g);
    int64_t m = g.nwin / (kWindowsPerCluster * (nres > 0 ? nres : 1));
    if (m > kMaxGroups) m = kMaxGroups;
    if (m > g.n) m = g.n;
    return m < 2 ? 1 : (int)m;
}

// The streams and events of one pipelined call, released when the call returns
// (CUDA frees them once the work queued on them has completed).
struct Pipeline {
    cudaStream_t score = nullptr, rest = nullptr;
    cudaEvent_t ev[64 + 3] = {};
    int nev = 0;
    ~Pipeline()
    {
        for (int i = 0; i < nev; ++i)
            if (ev[i]) cudaEventDestroy(ev[i]);
        if (score) cudaStreamDestroy(score);
        if (rest) cudaStreamDestroy(rest);
    }
    cudaError_t init(int nevents)
    {
        int least = 0, greatest = 0;
        cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&score, cudaStreamNonBlocking, greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&rest, cudaStreamNonBlocking, least);
        for (; e == cudaSuccess && nev < nevents; ++nev) e = cudaEventCreateWithFlags(&ev[nev], cudaEventDisableTiming);
        return e;
    }
};

}  // namespace

namespace kara {
// The argument checks and geometry of the entry points, for other sources of the library.
kara_status geo_from_args(const kara_cache *c, const kara_params *p, const kara_batch *b, Geo *g)
{
    return make_geo(c, p, b, g);
}
}  // namespace kara

Range::Range(const char *name) { nvtxRangePushA(name); }
Range::~Range() { nvtxRangePop(); }

extern "C" {

const char *kara_status_string(int status)
{
    switch (status) {
        case KARA_OK: return "KARA_OK";
        case KARA_EINVAL: return "KARA_EINVAL: argument or cached length out of range";
        case KARA_EUNSUPPORTED: return "KARA_EUNSUPPORTED: shape outside the supported set";
        case KARA_ENOBLOCKS: return "KARA_ENOBLOCKS: fresh-block list too short";
        case KARA_EDUPBLOCK: return "KARA_EDUPBLOCK: duplicate block id";
        case KARA_ECUDA: return "KARA_ECUDA: CUDA runtime error";
        case KARA_EBADBLOCK: return "KARA_EBADBLOCK: block id outside the pool";
        case KARA_ETIMEOUT: return "KARA_ETIMEOUT: bounded device wait ran out";
        case KARA_EWORKSPACE: return "KARA_EWORKSPACE: workspace missing or too small";
        default: return "KARA_UNKNOWN";
    }
}

int kara_version(void) { return 1; }

kara_status kara_plan(const kara_params *p, int32_t block_size, int32_t n, const int32_t *h_len,
                      int32_t bt_stride, int32_t *h_n_new, int32_t *h_n_old, int64_t *h_total_new,
                      int64_t *h_total_old)
{
    kara_status st = check_params(p);
    if (st != KARA_OK) return st;
    if (block_size < 1 || n < 0 || (n > 0 && !h_len)) return KARA_EINVAL;
    int64_t tn = 0, to = 0;
    for (int32_t s = 0; s < n; ++s) {
        const int64_t L = h_len[s];
        if (L < p->W || (L + block_size - 1) / block_size > bt_stride) return KARA_EINVAL;
        const int64_t ws = L - p->W, p0 = ws / block_size, Lnew = ws + p->R + p->B;
        const int32_t no = (int32_t)((L + block_size - 1) / block_size - p0);
        const int32_t nn = (int32_t)((Lnew + block_size - 1) / block_size - p0);
        if (h_n_new) h_n_new[s] = nn;
        if (h_n_old) h_n_old[s] = no;
        tn += nn;
        to += no;
    }
    if (h_total_new) *h_total_new = tn;
    if (h_total_old) *h_total_old = to;
    return KARA_OK;
}

size_t kara_workspace_size(const kara_cache *c, const kara_params *p, int32_t n)
{
    if (check_params(p) != KARA_OK || check_cache(c) != KARA_OK || n < 0) return 0;
    if ((c->num_q_heads / c->num_kv_heads) * p->W > kMaxGW) return 0;
    Geo g;
    memset(&g, 0, sizeof g);
    g.layers = c->num_layers;
    g.hkv = c->num_kv_heads;
    g.hq = c->num_q_heads;
    g.G = c->num_q_heads / c->num_kv_heads;
    g.D = c->head_dim;
    g.W = p->W;
    g.C = p->W - p->B;
    g.K = p->K;
    g.R = p->R;
    g.n = n;
    g.nwin = (int64_t)n * c->num_layers * c->num_kv_heads;
    return layout(g).total;
}

kara_status kara_score(const kara_cache *c, const kara_params *p, const kara_batch *b, float *scores,
                       void *ws, size_t ws_bytes, int32_t *err, kara_stream_t stream)
{
    const Range range("kara_score");
    Geo g;
    kara_status st = make_geo(c, p, b, &g);
    if (st != KARA_OK) return st;
    if (g.nwin == 0) return KARA_OK;
    if (!scores || !err) return KARA_EINVAL;
    const size_t need = score_scratch_bytes(g);
    if (need && (!ws || ws_bytes < need)) return KARA_EWORKSPACE;
    return cuda_status(launch_score(g, scores, ws, err, (cudaStream_t)stream));
}

kara_status kara_compact_queries(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                 const int32_t *kept, int32_t *err, kara_stream_t stream)
{
    const Range range("kara_compact_queries");
    kara_status st = check_params(p);
    if (st != KARA_OK) return st;
    st = check_cache(c);
    if (st != KARA_OK) return st;
    if (!b || b->n < 0) return KARA_EINVAL;
    if (b->n == 0) return KARA_OK;
    if (!b->len || !b->q || !kept || !err || !aligned16(b->q)) return KARA_EINVAL;
    if ((int64_t)b->n * c->num_layers * c->num_q_heads > 0x7fffffffLL) return KARA_EUNSUPPORTED;
    return cuda_status(launch_qring_compact(c, p, b, kept, err, (cudaStream_t)stream));
}

kara_status kara_append_queries(const kara_cache *c, const kara_params *p, const kara_batch *b, const void *q_new,
                                kara_stream_t stream)
{
    const Range range("kara_append_queries");
    kara_status st = check_params(p);
    if (st != KARA_OK) return st;
    st = check_cache(c);
    if (st != KARA_OK) return st;
    if (!b || b->n < 0) return KARA_EINVAL;
    if (b->n == 0) return KARA_OK;
    if (!b->len || !b->q || !q_new || !aligned16(b->q) || !aligned16(q_new)) return KARA_EINVAL;
    return cuda_status(launch_qring_append(c, p, b, q_new, (cudaStream_t)stream));
}

size_t kara_decode_workspace_size(const kara_cache *c, int32_t n, int32_t bt_stride)
{
    if (check_cache(c) != KARA_OK || n < 0 || bt_stride < 1) return 0;
    return decode_workspace_bytes(c, n, bt_stride);
}

kara_status kara_decode_attention(const kara_cache *c, int32_t layer, int32_t n, const int32_t *len,
                                  const int32_t *block_table, int32_t bt_stride, const void *q, float *out,
                                  void *ws, size_t ws_bytes, int32_t *err, kara_stream_t stream)
{
    const Range range("kara_decode_attention");
    kara_status st = check_cache(c);
    if (st != KARA_OK) return st;
    if (layer < 0 || layer >= c->num_layers || n < 0 || bt_stride < 1) return KARA_EINVAL;
    if (n == 0) return KARA_OK;
    if (!len || !block_table || !q || !out || !err) return KARA_EINVAL;
    if (!aligned16(q)) return KARA_EINVAL;
    if (n > 65535 || c->num_kv_heads > 65535 || c->num_q_heads > 65535) return KARA_EUNSUPPORTED;
    if ((int64_t)bt_stride * c->block_size > 0x7fffffffLL) return KARA_EUNSUPPORTED;
    if (decode_max_splits(bt_stride, c->block_size) > 65535) return KARA_EUNSUPPORTED;  // grid z
    if (!ws || ws_bytes < decode_workspace_bytes(c, n, bt_stride)) return KARA_EWORKSPACE;
    return cuda_status(launch_decode(c, layer, n, len, block_table, bt_stride, q, out, ws, err,
                                     (cudaStream_t)stream));
}

kara_status kara_select(const kara_params *p, int64_t n_windows, const float *scores, int32_t *cand,
                        int32_t *kept, kara_stream_t stream)
{
    const Range range("kara_select");
    kara_status st = check_params(p);
    if (st != KARA_OK) return st;
    if (n_windows < 0) return KARA_EINVAL;
    if (n_windows == 0) return KARA_OK;
    if (!scores || !kept) return KARA_EINVAL;
    if (n_windows > 0x7fffffffLL) return KARA_EUNSUPPORTED;
    return cuda_status(launch_select(n_windows, p->W - p->B, p->K, p->R, p->lambda, p->select_mode, p->chunk,
                                     scores, cand, kept, (cudaStream_t)stream));
}

kara_status kara_compact(const kara_cache *c, const kara_params *p, const kara_batch *b,
                         const int32_t *kept, const int32_t *fresh, int64_t n_fresh, int32_t *freed,
                         int32_t *new_len, int32_t *err, void *ws, size_t ws_bytes, kara_stream_t stream)
{
    const Range range("kara_compact");
    Geo g;
    kara_status st = make_geo(c, p, b, &g);
    if (st != KARA_OK) return st;
    if (g.n == 0) return KARA_OK;
    if (!kept || !new_len || !err || n_fresh < 0 || (n_fresh > 0 && !fresh) || !freed)
        return KARA_EINVAL;
    const WsLayout w = layout(g);
    if (!ws || ws_bytes < w.plan + align256((size_t)g.n * sizeof(SeqPlan))) return KARA_EWORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    SeqPlan *plan = at<SeqPlan>(ws, w.plan);
    cudaError_t e = launch_plan(g, n_fresh, plan, err, s);
    if (e == cudaSuccess) e = launch_compact(g, plan, kept, fresh, n_fresh, err, s);
    if (e == cudaSuccess) e = launch_commit(g, plan, fresh, freed, new_len, b->block_table, err, s);
    return cuda_status(e);
}

kara_status kara_compress_batch(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                const int32_t *fresh, int64_t n_fresh, int32_t *freed, int32_t *new_len,
                                float *scores_out, int32_t *cand_out, int32_t *kept_out, void *ws,
                                size_t ws_bytes, int32_t *err, kara_stream_t stream,
                                void *const *phase_events)
{
    const Range range("kara_compress_batch");
    Geo g;
    kara_status st = make_geo(c, p, b, &g);
    if (st != KARA_OK) return st;
    if (g.n == 0) return KARA_OK;
    if (!new_len || !err || n_fresh < 0 || (n_fresh > 0 && !fresh) || !freed) return KARA_EINVAL;
    if (g.nwin > 0x7fffffffLL) return KARA_EUNSUPPORTED;
    const WsLayout w = layout(g);
    if (!ws || ws_bytes < w.total) return KARA_EWORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    SeqPlan *plan = at<SeqPlan>(ws, w.plan);
    float *scores = scores_out ? scores_out : at<float>(ws, w.scores);
    int32_t *cand = cand_out ? cand_out : at<int32_t>(ws, w.cand);
    int32_t *kept = kept_out ? kept_out : at<int32_t>(ws, w.kept);
    auto mark = [&](int i) -> cudaError_t {
        return phase_events ? cudaEventRecord((cudaEvent_t)phase_events[i], s) : cudaSuccess;
    };
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return KARA_ECUDA;
    const int m = cap == cudaStreamCaptureStatusNone ? batch_groups(g) : 1;
    if (m > 1) {
        // groups of sequences: scoring on a high-priority stream, selection and
        // copy of each scored group on a low-priority one, both forked from and
        // joined back to `stream`
        Pipeline pl;
        uint8_t *scratch = at<uint8_t>(ws, w.scratch);
        cudaError_t e = pl.init(m + 3);
        if (e == cudaSuccess) e = mark(0);
        if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int32_t), s);
        if (e == cudaSuccess) e = launch_plan(g, n_fresh, plan, err, s);
        if (e == cudaSuccess) e = launch_fresh_check(g, plan, fresh, n_fresh, err, s);
        if (e == cudaSuccess) e = mark(1);
        if (e == cudaSuccess) e = cudaEventRecord(pl.ev[0], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(pl.score, pl.ev[0], 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(pl.rest, pl.ev[0], 0);
        const bool forked = e == cudaSuccess;
        const int64_t wps = (int64_t)g.layers * g.hkv;  // windows per sequence
        for (int i = 0; i < m && e == cudaSuccess; ++i) {
            const int s0 = (int)((int64_t)i * g.n / m), s1 = (int)((int64_t)(i + 1) * g.n / m);
            const Geo gi = sub_batch(g, s0, s1);
            const int64_t u0 = s0 * wps;
            e = launch_score(gi, scores + u0 * g.C, scratch + u0, err, pl.score);
            if (e == cudaSuccess) e = cudaEventRecord(pl.ev[1 + i], pl.score);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(pl.rest, pl.ev[1 + i], 0);
            if (e == cudaSuccess)
                e = launch_select(gi.nwin, g.C, g.K, g.R, g.lambda, p->select_mode, p->chunk, scores + u0 * g.C,
                                  cand + u0 * g.K, kept + u0 * g.R, pl.rest);
            if (e == cudaSuccess) e = launch_kept_copy(gi, plan + s0, kept + u0 * g.R, fresh, n_fresh, err, pl.rest);
        }
        if (e == cudaSuccess && phase_events) e = cudaEventRecord((cudaEvent_t)phase_events[2], pl.score);
        if (forked) {
            // both streams join `stream` even after a failed launch, so nothing the
            // call queued is still running when later work on `stream` starts
            cudaError_t j = cudaEventRecord(pl.ev[1 + m], pl.rest);  // after every group (rest waited on each)
            if (j == cudaSuccess) j = cudaStreamWaitEvent(s, pl.ev[1 + m], 0);
            if (j == cudaSuccess) j = cudaEventRecord(pl.ev[2 + m], pl.score);
            if (j == cudaSuccess) j = cudaStreamWaitEvent(s, pl.ev[2 + m], 0);
            if (e == cudaSuccess) e = j;
        }
        if (e == cudaSuccess) e = mark(3);
        if (e == cudaSuccess) e = launch_commit(g, plan, fresh, freed, new_len, b->block_table, err, s);
        if (e == cudaSuccess) e = mark(4);
        return cuda_status(e);
    }
    cudaError_t e = mark(0);
    if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = launch_plan(g, n_fresh, plan, err, s);
    if (e == cudaSuccess) e = mark(1);
    if (e == cudaSuccess) e = launch_score(g, scores, at<void>(ws, w.scratch), err, s);
    if (e == cudaSuccess) e = mark(2);
    if (e == cudaSuccess) e = launch_select(g.nwin, g.C, g.K, g.R, g.lambda, p->select_mode, p->chunk, scores, cand,
                                            kept, s);
    if (e == cudaSuccess) e = mark(3);
    if (e == cudaSuccess) e = launch_compact(g, plan, kept, fresh, n_fresh, err, s);
    if (e == cudaSuccess) e = launch_commit(g, plan, fresh, freed, new_len, b->block_table, err, s);
    if (e == cudaSuccess) e = mark(4);
    return cuda_status(e);
}

int32_t kara_batch_groups(const kara_cache *c, const kara_params *p, const kara_batch *b)
{
    Geo g;
    const kara_status st = make_geo(c, p, b, &g);
    if (st != KARA_OK) return (int32_t)st;
    return batch_groups(g);
}

kara_status kara_get_error(const int32_t *err, kara_stream_t stream)
{
    if (!err) return KARA_EINVAL;
    int32_t h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, err, sizeof h, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return KARA_ECUDA;
    return (kara_status)h;
}

}  // extern "C"
