// The window-query ring: the queries that score a window, kept on the device
// and compacted together with K and V.
//
// The pages do not say where window queries live (the gist.science summary
// of Kara, section 1 "Mechanism": the queries of all W window tokens score the
// window).  Here each (sequence, layer, query head) keeps the queries of its
// last W positions in a ring of W rows: the query of logical position x is in
// row x mod W.  The scores do not depend on the order of the query rows (each
// row's softmax is its own and the rows are summed), so the bidirectional
// scorer reads the ring as it stands.  When a step compacts K and V, the
// queries of the kept rows and of the protected buffer move to the same new
// positions:
//     row (ws + r) mod W     <- row (ws + kept[r]) mod W,  r < R
//     row (ws + R + b) mod W <- row (L - B + b) mod W,     b < B
#include "kara_common.cuh"

namespace kara {
namespace {

constexpr int kQThreads = 128;
constexpr int kQChunk = 64;  // rows staged per round

struct QArgs {
    uint16_t *ring;       // [n][layers][hq][W][D]
    const uint16_t *q_new;  // [n][layers][hq][D] (append)
    const int32_t *len;
    const int32_t *kept;  // [n][layers][hkv][R]
    int32_t *err;
    int32_t n, layers, hq, hkv, G, W, B, R;
};

// One CTA per (sequence, layer, query head).  New window index r takes its
// row from source index src(r) = kept[r] (r < R) or W - B + (r - R).  kept is
// strictly increasing, so src(r) >= r and the sources increase with r: moving
// rows in increasing r, a chunk's sources are never destinations of earlier
// chunks, and staging the chunk's sources in shared memory before writing
// covers the overlap inside the chunk.  The move is therefore safe in place.
template <int D>
__global__ void __launch_bounds__(kQThreads) qring_compact_kernel(const QArgs a)
{
    constexpr int VPR = D / 8;  // 16-byte vectors per row
    __shared__ uint4 buf[kQChunk * VPR];
    __shared__ int bad;
    // a failed step commits nothing, queries included (read once, so that the
    // whole CTA takes the same branch)
    if (threadIdx.x == 0) bad = *(volatile int32_t *)a.err != 0;
    __syncthreads();
    if (bad) return;
    __syncthreads();
    const int h = blockIdx.x % a.hq;
    const int l = (blockIdx.x / a.hq) % a.layers;
    const int s = blockIdx.x / (a.hq * a.layers);
    const int32_t L = a.len[s];
    if (L < a.W) return;  // the step has recorded the error already
    const int W = a.W, R = a.R, C = a.W - a.B;
    const int ws_mod = (L - W) % W;
    const int32_t *kp = a.kept + (((int64_t)s * a.layers + l) * a.hkv + h / a.G) * R;
    uint4 *ring = reinterpret_cast<uint4 *>(a.ring + (((int64_t)s * a.layers + l) * a.hq + h) * W * D);

    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    // kept must be the step's output: strictly increasing in [0, C); a window
    // whose row is not is reported and left as it is
    for (int r = threadIdx.x; r < R; r += kQThreads) {
        const int32_t x = kp[r];
        if (x < r || x >= C || (r > 0 && kp[r - 1] >= x)) bad = 1;
    }
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) set_err(a.err, KARA_EINVAL);
        return;
    }
    const int nrows = R + a.B;
    for (int r0 = 0; r0 < nrows; r0 += kQChunk) {
        const int nr = min(kQChunk, nrows - r0);
        for (int i = threadIdx.x; i < nr * VPR; i += kQThreads) {
            const int r = r0 + i / VPR;
            const int src = r < R ? kp[r] : W - a.B + (r - R);
            const int row = ws_mod + src >= W ? ws_mod + src - W : ws_mod + src;
            buf[i] = ring[(int64_t)row * VPR + i % VPR];
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nr * VPR; i += kQThreads) {
            const int r = r0 + i / VPR;
            const int row = ws_mod + r >= W ? ws_mod + r - W : ws_mod + r;
            ring[(int64_t)row * VPR + i % VPR] = buf[i];
        }
        __syncthreads();
    }
}

// q_new[s][l][h] -> ring row len[s] mod W, one 16-byte vector per thread.
template <int D>
__global__ void qring_append_kernel(const QArgs a)
{
    constexpr int VPR = D / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (int64_t)a.n * a.layers * a.hq * VPR;
    if (i >= total) return;
    const int64_t head = i / VPR;  // (s, l, h)
    const int s = (int)(head / ((int64_t)a.layers * a.hq));
    const int32_t L = a.len[s];
    if (L < 0) return;
    const int row = L % a.W;
    reinterpret_cast<uint4 *>(a.ring)[(head * a.W + row) * VPR + i % VPR] =
        reinterpret_cast<const uint4 *>(a.q_new)[i];
}

QArgs qargs(const kara_cache *c, const kara_params *p, const kara_batch *b)
{
    QArgs a;
    a.ring = static_cast<uint16_t *>(const_cast<void *>(b->q));
    a.q_new = nullptr;
    a.len = b->len;
    a.kept = nullptr;
    a.err = nullptr;
    a.n = b->n;
    a.layers = c->num_layers;
    a.hq = c->num_q_heads;
    a.hkv = c->num_kv_heads;
    a.G = c->num_q_heads / c->num_kv_heads;
    a.W = p->W;
    a.B = p->B;
    a.R = p->R;
    return a;
}

}  // namespace

cudaError_t launch_qring_compact(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                 const int32_t *kept, int32_t *err, cudaStream_t st)
{
    QArgs a = qargs(c, p, b);
    a.kept = kept;
    a.err = err;
    const int64_t grid = (int64_t)a.n * a.layers * a.hq;
    if (grid == 0) return cudaSuccess;
    if (c->head_dim == 128)
        qring_compact_kernel<128><<<(unsigned)grid, kQThreads, 0, st>>>(a);
    else
        qring_compact_kernel<64><<<(unsigned)grid, kQThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_qring_append(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                const void *q_new, cudaStream_t st)
{
    QArgs a = qargs(c, p, b);
    a.q_new = static_cast<const uint16_t *>(q_new);
    const int64_t total = (int64_t)a.n * a.layers * a.hq * (c->head_dim / 8);
    if (total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((total + 255) / 256);
    if (c->head_dim == 128)
        qring_append_kernel<128><<<blocks, 256, 0, st>>>(a);
    else
        qring_append_kernel<64><<<blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kara
