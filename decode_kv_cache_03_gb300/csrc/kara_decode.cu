// Decode attention over the paged cache: the reader of the block tables the
// compression step rewrites.
//
// Follows the gist.science summary of Kara (arXiv 2607.01237), section
// "3. KvLLM Framework and Periodic Compression": Kara is adapted to
// PagedAttention, and the blocks a compression frees let more sequences
// decode.  One decode query per sequence and query head h attends to every
// cached key x < L of its sequence in one layer (KV head g = h / G):
//     o_h = sum_x softmax_x(<q_h, k_x> / sqrt(D)) v_x
// with K and V read through the block table.  Logits, softmax and sums are
// fp32 (logits in the log2 domain); the output is fp32.
//
// The work is HBM-bound (about 2.5 FLOP per byte of K and V), so it runs on
// the CUDA cores.  Flash-decoding layout: one CTA per (sequence, KV head,
// split of kSplit keys).  A producer warp streams the split's K blocks, then
// its V blocks, into a ring of shared-memory stages with the bulk-copy engine
// (each (block, KV head) of a pool is one contiguous 16 x D bf16 region), so
// many blocks are in flight per SM without holding registers.  Four consumer
// warps take one block each: logits with 8 lanes per key and packed fp32
// pairs, then the softmax of the split in shared memory, then the weighted
// sum of V.  A second kernel combines the splits of each (sequence, head) in
// a fixed order, so the result is deterministic.
#include "kara_common.cuh"
#include "kara_sm100.cuh"

namespace kara {
namespace {

constexpr int kSplit = 1024;        // keys per CTA
constexpr int kBlk = 16;            // tokens per cache block (the supported block size)
constexpr int kBlocks = kSplit / kBlk;
constexpr int kNC = 4;              // consumer warps
constexpr int kDecThreads = 32 * (1 + kNC);
constexpr int kStages = 12;         // ring of (block, head) slices in flight
constexpr uint64_t kDecTimeoutNs = 1000000000ull;  // 1 s: a stage normally lands in microseconds
// Blocks go to the consumer warps round-robin and stage waits are by phase
// parity, which tells only two neighbouring phases apart: a warp may wait for
// use j of a stage only after it has seen use j - kStages complete, so both
// uses must be its own.
static_assert(kStages % kNC == 0, "each stage is reused by the same consumer warp");

struct DecodeArgs {
    const uint16_t *k, *v;
    int64_t layer_off, block_stride, head_stride;
    int32_t num_blocks, hkv, hq, G, bs;
    const int32_t *len;
    const int32_t *bt;
    int32_t bt_stride, n, max_splits;
    const uint16_t *q;   // [n][hq][D]
    float *part;         // [n][hq][max_splits][D]
    float2 *stat;        // [n][hq][max_splits]: (max, sum) in the log2 domain
    float *out;          // [n][hq][D]
    float scale2;        // log2(e) / sqrt(D)
    int32_t stall;       // debug: the producer issues nothing (see debug_stall)
    uint64_t wait_ns;    // limit of the waits on progress
};

__device__ __forceinline__ bool length_ok(const DecodeArgs &a, int32_t L)
{
    return L >= 1 && ((int64_t)L + a.bs - 1) / a.bs <= a.bt_stride;
}

// Barriers and per-split tables of one CTA (after the ring and the logits in
// dynamic shared memory).
struct DecShared {
    uint64_t full[kStages], empty[kStages];
    int32_t blk[kBlocks];   // physical ids of the split's blocks
    int32_t bad[kStages];   // the stage's block id was outside the pool: read as zeros
    float2 st_m[8];         // per head: (max, sum) of the split in the log2 domain
    int32_t abort;
};

// Bounded wait on phase `parity` of `bar`.  Gives up after limit_ns, or when
// another warp of the CTA gave up, recording KARA_ETIMEOUT.
__device__ bool dwait(uint32_t bar, uint32_t parity, DecShared *sh, int32_t *err, uint64_t limit_ns,
                      bool honour_abort = true)
{
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u) {
            if (honour_abort && *(volatile int32_t *)&sh->abort) return false;
            const uint64_t now = ptx::globaltimer();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > limit_ns) {
                set_err(err, KARA_ETIMEOUT);
                *(volatile int32_t *)&sh->abort = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float fold2(uint64_t r)
{
    float lo, hi;
    ptx::unpack2(r, lo, hi);
    return lo + hi;
}

// Weighted sum of one V block into acc: lane owns dims [lane*2*VW, +2*VW),
// tokens taken in pairs so that one packed FMA uses the weights of two
// adjacent tokens, (p_t, p_t+1) * (v_t, v_t+1).  MASK: the block is the last
// one of the split and holds tmax < 16 valid rows; rows past it are zeroed
// (their bytes are whatever the block held) and their weights are 0.
template <int D, int G, bool MASK>
__device__ __forceinline__ void v_block(const uint8_t *blkp, const float *wrow, int tmax, int lane,
                                        uint64_t (&acc)[G][2 * (D / 64)])
{
    constexpr int VW = D / 64;  // 32-bit words (bf16 pairs) per row per lane
#pragma unroll
    for (int t = 0; t < kBlk; t += 2) {
        if (MASK && t >= tmax) break;
        uint32_t w0[VW], w1[VW];
        if constexpr (VW == 2) {
            const uint2 a = *reinterpret_cast<const uint2 *>(blkp + t * D * 2 + lane * 8);
            const uint2 b = *reinterpret_cast<const uint2 *>(blkp + (t + 1) * D * 2 + lane * 8);
            w0[0] = a.x, w0[1] = a.y, w1[0] = b.x, w1[1] = b.y;
        } else {
            w0[0] = *reinterpret_cast<const uint32_t *>(blkp + t * D * 2 + lane * 4);
            w1[0] = *reinterpret_cast<const uint32_t *>(blkp + (t + 1) * D * 2 + lane * 4);
        }
        if (MASK && t + 1 >= tmax)
#pragma unroll
            for (int e = 0; e < VW; ++e) w1[e] = 0u;
        uint64_t vp[2 * VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) {
            vp[2 * e] = ptx::pack2(lo_f(w0[e]), lo_f(w1[e]));
            vp[2 * e + 1] = ptx::pack2(hi_f(w0[e]), hi_f(w1[e]));
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const uint64_t pp = *reinterpret_cast<const uint64_t *>(wrow + h * kSplit + t);
#pragma unroll
            for (int d = 0; d < 2 * VW; ++d) acc[h][d] = ptx::fma2(pp, vp[d], acc[h][d]);
        }
    }
}

// Dynamic shared memory: ring[kStages][16][D] bf16, logit[G][kSplit] fp32
// (logits, then weights, then the consumers' partial outputs), DecShared.
// Three CTAs per SM (128 registers a thread) except for the widest groups,
// whose queries take too many registers for that.
template <int D, int G>
constexpr int dec_min_blocks() { return D == 128 && G >= 6 ? 2 : 3; }

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, dec_min_blocks<D, G>()) decode_split_kernel(const DecodeArgs a, int32_t *err)
{
    constexpr int BB = kBlk * D * 2;  // bytes of one (block, head) slice
    constexpr int NCH = D / 64;       // 8-dim chunks per lane in the logits (dims c*64 + sub*8 ..)
    constexpr int VW = D / 64;
    static_assert(G <= 8, "heads per group");
    static_assert(kNC * D <= kSplit, "partial outputs fit in the logit area");
    extern __shared__ __align__(128) uint8_t dsm[];
    uint8_t *ring = dsm;
    float *logit = reinterpret_cast<float *>(dsm + kStages * BB);  // [G][kSplit]
    DecShared *sh = reinterpret_cast<DecShared *>(logit + G * kSplit);

    const int sp = blockIdx.z, g = blockIdx.x, s = blockIdx.y;
    const int32_t L = a.len[s];
    if (!length_ok(a, L)) {
        if (sp == 0 && g == 0 && threadIdx.x == 0) set_err(err, KARA_EINVAL);
        return;
    }
    const int32_t k0 = sp * kSplit;
    if (k0 >= L) return;
    const int nk = min(kSplit, L - k0);
    const int nb = (nk + kBlk - 1) / kBlk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i < nb; i += kDecThreads) sh->blk[i] = a.bt[(int64_t)s * a.bt_stride + k0 / kBlk + i];
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(ptx::smem_u32(&sh->full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&sh->empty[i]), 1);
        }
        sh->abort = 0;
        ptx::fence_mbarrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------- producer: K blocks 0..nb-1, then V blocks --------------
        if (lane == 0) {
            const int64_t head_off = a.layer_off + (int64_t)g * a.head_stride;
            int issued = 0;
            for (int j = 0; j < (a.stall ? 0 : 2 * nb); ++j) {
                const int st = j % kStages;
                if (!dwait(ptx::smem_u32(&sh->empty[st]), ((j / kStages) & 1) ^ 1, sh, err, a.wait_ns)) break;
                const int32_t blk = sh->blk[j < nb ? j : j - nb];
                const uint32_t fb = ptx::smem_u32(&sh->full[st]);
                if (blk < 0 || blk >= a.num_blocks) {
                    set_err(err, KARA_EBADBLOCK);
                    sh->bad[st] = 1;
                    ptx::mbar_arrive(fb);
                } else {
                    sh->bad[st] = 0;
                    ptx::mbar_arrive_expect_tx(fb, BB);
                    ptx::bulk_load(ptx::smem_u32(ring + st * BB), (j < nb ? a.k : a.v) + head_off + (int64_t)blk * a.block_stride,
                                   BB, fb);
                }
                issued = j + 1;
            }
            // every copy issued has landed before the CTA's shared memory is released
            for (int j = max(0, issued - kStages); j < issued; ++j)
                dwait(ptx::smem_u32(&sh->full[j % kStages]), (j / kStages) & 1, sh, err, kDecTimeoutNs, false);
        }
        return;
    }

    // ---------------- consumers ----------------------------------------------------
    const int cw = warp - 1, grp = lane >> 3, sub = lane & 7;
    const int ctid = threadIdx.x - 32;

    // this lane's dims of the G queries (c*64 + sub*8 + [0, 8)), pre-scaled into
    // the log2 domain, as (even, odd) pairs
    uint64_t qv[G][NCH][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const uint4 r = __ldg(reinterpret_cast<const uint4 *>(a.q + ((int64_t)s * a.hq + g * G + h) * D + c * 64 + sub * 8));
            const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) qv[h][c][e] = ptx::pack2(lo_f(w[e]) * a.scale2, hi_f(w[e]) * a.scale2);
        }

    // ---- logits: lane group grp takes tokens grp + 4k of the block, 8 lanes per token
    for (int i = cw; i < nb; i += kNC) {
        const int st = i % kStages;
        if (!dwait(ptx::smem_u32(&sh->full[st]), (i / kStages) & 1, sh, err, a.wait_ns)) break;
        const bool bad = sh->bad[st] != 0;
        const uint8_t *blkp = ring + st * BB;
        float dot[4][G];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int t = grp + 4 * k;
            uint64_t acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = 0ull;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const uint4 r = *reinterpret_cast<const uint4 *>(blkp + t * D * 2 + c * 128 + sub * 16);
                const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint64_t kp = ptx::pack2(lo_f(w[e]), hi_f(w[e]));
#pragma unroll
                    for (int h = 0; h < G; ++h) acc[h] = ptx::fma2(qv[h][c][e], kp, acc[h]);
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) dot[k][h] = fold2(acc[h]);
        }
        // the block's bytes are in registers: hand the stage back
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sh->empty[st]));
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int o = 4; o > 0; o >>= 1) dot[k][h] += __shfl_xor_sync(0xffffffffu, dot[k][h], o);
        // lane sub = k of the group writes token grp + 4k (a zero row gives logit 0)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int x = i * kBlk + grp + 4 * k;
            if (sub == k && x < nk)
#pragma unroll
                for (int h = 0; h < G; ++h) logit[h * kSplit + x] = bad ? 0.f : dot[k][h];
        }
    }
    ptx::named_barrier(1, kNC * 32);

    // ---- softmax of each head over the split (warp cw: heads cw, cw + kNC) -------
    for (int h = cw; h < G; h += kNC) {
        float *lr = logit + h * kSplit;
        float m = -INFINITY;
        for (int x = lane; x < nk; x += 32) m = fmaxf(m, lr[x]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float z = 0.f;
        for (int x = lane; x < nk; x += 32) {
            const float p = ptx::ex2(lr[x] - m);
            lr[x] = p;
            z += p;
        }
        for (int x = nk + lane; x < nb * kBlk; x += 32) lr[x] = 0.f;  // rows past the end weigh 0
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        if (lane == 0) sh->st_m[h] = make_float2(m, z);
    }
    ptx::named_barrier(1, kNC * 32);

    // ---- weighted sum of V ----------------------------------------------------------
    uint64_t acc[G][2 * VW];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int d = 0; d < 2 * VW; ++d) acc[h][d] = 0ull;
    for (int i = cw; i < nb; i += kNC) {
        const int j = nb + i, st = j % kStages;
        if (!dwait(ptx::smem_u32(&sh->full[st]), (j / kStages) & 1, sh, err, a.wait_ns)) break;
        if (sh->bad[st] == 0) {
            const int tmax = min(kBlk, nk - i * kBlk);
            if (tmax == kBlk)
                v_block<D, G, false>(ring + st * BB, logit + i * kBlk, tmax, lane, acc);
            else
                v_block<D, G, true>(ring + st * BB, logit + i * kBlk, tmax, lane, acc);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sh->empty[st]));
    }
    // every consumer is done with the weights: the logit area takes the partial
    // outputs red[kNC][G][D], summed below over the warps in a fixed order
    ptx::named_barrier(1, kNC * 32);
    float *red = logit;
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int d = 0; d < 2 * VW; ++d) red[(cw * G + h) * D + lane * 2 * VW + d] = fold2(acc[h][d]);
    ptx::named_barrier(1, kNC * 32);
    for (int x = ctid; x < G * D; x += kNC * 32) {
        const int h = x / D, d = x % D;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kNC; ++w) v += red[(w * G + h) * D + d];
        const int64_t idx = ((int64_t)s * a.hq + g * G + h) * a.max_splits + sp;
        a.part[idx * D + d] = v;
        if (d == 0) a.stat[idx] = sh->st_m[h];
    }
}

// out[s][h] = sum_sp part * 2^(m_sp - M) / sum_sp z_sp * 2^(m_sp - M), splits in order.
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeArgs a)
{
    const int h = blockIdx.x, s = blockIdx.y, d = threadIdx.x;
    const int32_t L = a.len[s];
    float *o = a.out + ((int64_t)s * a.hq + h) * D;
    if (!length_ok(a, L)) {
        o[d] = 0.f;
        return;
    }
    const int nsp = (L + kSplit - 1) / kSplit;
    const int64_t base = ((int64_t)s * a.hq + h) * a.max_splits;
    float M = -INFINITY;
    for (int sp = 0; sp < nsp; ++sp) M = fmaxf(M, a.stat[base + sp].x);
    float den = 0.f, num = 0.f;
    for (int sp = 0; sp < nsp; ++sp) {
        const float2 st = a.stat[base + sp];
        const float w = exp2f(st.x - M);
        den = fmaf(st.y, w, den);
        num = fmaf(a.part[(base + sp) * D + d], w, num);
    }
    o[d] = num / den;
}

template <int D, int G>
cudaError_t launch_split_g(const DecodeArgs &a, dim3 grid, int32_t *err, cudaStream_t st)
{
    const size_t smem = (size_t)kStages * kBlk * D * 2 + sizeof(float) * G * kSplit + sizeof(DecShared);
    auto kern = decode_split_kernel<D, G>;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kDecThreads, smem, st>>>(a, err);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_split(const DecodeArgs &a, dim3 grid, int32_t *err, cudaStream_t st)
{
    switch (a.G) {
        case 1: return launch_split_g<D, 1>(a, grid, err, st);
        case 2: return launch_split_g<D, 2>(a, grid, err, st);
        case 3: return launch_split_g<D, 3>(a, grid, err, st);
        case 4: return launch_split_g<D, 4>(a, grid, err, st);
        case 5: return launch_split_g<D, 5>(a, grid, err, st);
        case 6: return launch_split_g<D, 6>(a, grid, err, st);
        case 7: return launch_split_g<D, 7>(a, grid, err, st);
        case 8: return launch_split_g<D, 8>(a, grid, err, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int decode_max_splits(int32_t bt_stride, int32_t block_size)
{
    return (int)(((int64_t)bt_stride * block_size + kSplit - 1) / kSplit);
}

cudaError_t launch_decode(const kara_cache *c, int32_t layer, int32_t n, const int32_t *len, const int32_t *bt,
                          int32_t bt_stride, const void *q, float *out, void *ws, int32_t *err, cudaStream_t st)
{
    if (n == 0) return cudaSuccess;
    DecodeArgs a;
    a.k = static_cast<const uint16_t *>(c->k);
    a.v = static_cast<const uint16_t *>(c->v);
    a.layer_off = (int64_t)layer * c->layer_stride;
    a.block_stride = c->block_stride;
    a.head_stride = c->head_stride;
    a.num_blocks = c->num_blocks;
    a.hkv = c->num_kv_heads;
    a.hq = c->num_q_heads;
    a.G = c->num_q_heads / c->num_kv_heads;
    a.bs = c->block_size;
    a.len = len;
    a.bt = bt;
    a.bt_stride = bt_stride;
    a.n = n;
    a.max_splits = decode_max_splits(bt_stride, c->block_size);
    a.q = static_cast<const uint16_t *>(q);
    const size_t npart = (size_t)n * a.hq * a.max_splits;
    a.part = static_cast<float *>(ws);
    a.stat = reinterpret_cast<float2 *>(static_cast<char *>(ws) + align256(npart * c->head_dim * sizeof(float)));
    a.out = out;
    a.scale2 = 1.4426950408889634f / sqrtf((float)c->head_dim);
    const Stall dbg = debug_stall(kDecTimeoutNs);
    a.stall = dbg.on;
    a.wait_ns = dbg.wait_ns;
    // split-major: CTAs past a short sequence's end (they exit at once) come last,
    // where they take slots the grid's tail leaves idle anyway
    const dim3 grid((unsigned)a.hkv, (unsigned)n, (unsigned)a.max_splits);
    cudaError_t e = c->head_dim == 128 ? launch_split<128>(a, grid, err, st) : launch_split<64>(a, grid, err, st);
    if (e != cudaSuccess) return e;
    if (c->head_dim == 128)
        decode_combine_kernel<128><<<dim3((unsigned)a.hq, (unsigned)n), 128, 0, st>>>(a);
    else
        decode_combine_kernel<64><<<dim3((unsigned)a.hq, (unsigned)n), 64, 0, st>>>(a);
    return cudaGetLastError();
}

size_t decode_workspace_bytes(const kara_cache *c, int32_t n, int32_t bt_stride)
{
    const size_t npart = (size_t)n * c->num_q_heads * decode_max_splits(bt_stride, c->block_size);
    return align256(npart * c->head_dim * sizeof(float)) + align256(npart * sizeof(float2));
}

}  // namespace kara
