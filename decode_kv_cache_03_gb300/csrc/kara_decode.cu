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
// split of kSplit keys) streams its keys twice -- K for the logits, V for the
// weighted sum -- with 16 lanes per key row (16-byte loads) and four keys
// per lane in flight; a second kernel combines the splits of each (sequence, head)
// in a fixed order, so the result is deterministic.
#include "kara_common.cuh"

namespace kara {
namespace {

constexpr int kSplit = 1024;        // keys per CTA
constexpr int kDecThreads = 256;    // 8 warps
constexpr int kLanesPerKey = 16;

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
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ bool length_ok(const DecodeArgs &a, int32_t L)
{
    return L >= 1 && ((int64_t)L + a.bs - 1) / a.bs <= a.bt_stride;
}

// Elements [sub*DL, sub*DL + DL) of the row of logical position x of sequence
// s, KV head g; nullptr for a block id outside the pool (recorded in err).
template <int D, int DL>
__device__ __forceinline__ const uint16_t *row_ptr(const DecodeArgs &a, const uint16_t *pool, int s, int g,
                                                   int32_t x, int sub, int32_t *err)
{
    const int32_t blk = a.bt[(int64_t)s * a.bt_stride + x / a.bs];
    if (blk < 0 || blk >= a.num_blocks) {
        set_err(err, KARA_EBADBLOCK);
        return nullptr;
    }
    return pool + a.layer_off + (int64_t)blk * a.block_stride + (int64_t)g * a.head_stride +
           (int64_t)(x % a.bs) * D + sub * DL;
}

// DL (4, 8 or 16) bf16 of a row at p, as ceil(DL/8) uint4 (a 4-element slice
// fills the first half of r[0]).
template <int DL>
__device__ __forceinline__ void load_slice(const uint16_t *p, uint4 (&r)[(DL + 7) / 8])
{
    if constexpr (DL == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        r[0] = make_uint4(u.x, u.y, 0u, 0u);
    } else {
#pragma unroll
        for (int i = 0; i < DL / 8; ++i) r[i] = __ldg(reinterpret_cast<const uint4 *>(p) + i);
    }
}

// Dynamic shared memory: p[G][kSplit] (logits, then weights) and red[8][G][D].
template <int D, int G>
__global__ void __launch_bounds__(kDecThreads) decode_split_kernel(const DecodeArgs a, int32_t *err)
{
    constexpr int DL = D / kLanesPerKey;  // dims per lane: 8 (D = 128) or 4 (D = 64)
    constexpr int NV = (DL + 7) / 8;      // uint4 per lane per row
    constexpr int E = DL < 8 ? DL : 8;    // valid elements per uint4
    constexpr int KPW = 32 / kLanesPerKey;  // keys per warp and round
    constexpr int kUnroll = 4;              // keys per lane in flight (more costs occupancy)
    static_assert(DL == 8 || DL == 4, "head dim");
    static_assert(G <= kDecThreads / 32, "one warp per head in the softmax step");
    extern __shared__ float dsm[];
    float(*logit)[kSplit] = reinterpret_cast<float(*)[kSplit]>(dsm);
    float(*red)[G][D] = reinterpret_cast<float(*)[G][D]>(dsm + G * kSplit);
    __shared__ float2 st_m[G];

    const int sp = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int32_t L = a.len[s];
    if (!length_ok(a, L)) {
        if (sp == 0 && g == 0 && threadIdx.x == 0) set_err(err, KARA_EINVAL);
        return;
    }
    const int32_t k0 = sp * kSplit;
    if (k0 >= L) return;
    const int nk = min(kSplit, L - k0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane / kLanesPerKey, sub = lane % kLanesPerKey;  // key slot in the warp, dim slice

    // this lane's slice of the G queries, pre-scaled into the log2 domain
    float qv[G][DL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        uint4 r[NV];
        load_slice<DL>(a.q + ((int64_t)s * a.hq + g * G + h) * D + sub * DL, r);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float f[8];
            bf16x8_to_f32(r[i], f);
#pragma unroll
            for (int e = 0; e < E; ++e) qv[h][8 * i + e] = f[e] * a.scale2;
        }
    }

    // ---- logits: 16 lanes per key, kUnroll keys per lane in flight ---------
    constexpr int kKeysPerRound = (kDecThreads / 32) * KPW;  // 16
    for (int base = 0; base < nk; base += kKeysPerRound * kUnroll) {
        uint4 raw[kUnroll][NV];
#pragma unroll
        for (int uu = 0; uu < kUnroll; ++uu) {
            const int kk = base + uu * kKeysPerRound + warp * KPW + half;
#pragma unroll
            for (int i = 0; i < NV; ++i) raw[uu][i] = make_uint4(0u, 0u, 0u, 0u);
            if (kk < nk) {
                const uint16_t *r = row_ptr<D, DL>(a, a.k, s, g, k0 + kk, sub, err);
                if (r) load_slice<DL>(r, raw[uu]);
            }
        }
#pragma unroll
        for (int uu = 0; uu < kUnroll; ++uu) {
            const int kk = base + uu * kKeysPerRound + warp * KPW + half;
            float dot[G];
#pragma unroll
            for (int h = 0; h < G; ++h) dot[h] = 0.f;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                float kf[8];
                bf16x8_to_f32(raw[uu][i], kf);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < E; ++e) dot[h] = fmaf(qv[h][8 * i + e], kf[e], dot[h]);
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int o = kLanesPerKey / 2; o > 0; o >>= 1) dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], o);
            if (sub == 0 && kk < nk)
#pragma unroll
                for (int h = 0; h < G; ++h) logit[h][kk] = dot[h];
        }
    }
    __syncthreads();

    // ---- softmax of each head over this split: warp h --------------------------
    if (warp < G) {
        float m = -INFINITY;
        for (int kk = lane; kk < nk; kk += 32) m = fmaxf(m, logit[warp][kk]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float z = 0.f;
        for (int kk = lane; kk < nk; kk += 32) {
            const float p = exp2f(logit[warp][kk] - m);
            logit[warp][kk] = p;
            z += p;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        if (lane == 0) st_m[warp] = make_float2(m, z);
    }
    __syncthreads();

    // ---- weighted sum of V ---------------------------------------------------
    float acc[G][DL];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[h][e] = 0.f;
    for (int base = 0; base < nk; base += kKeysPerRound * kUnroll) {
        uint4 raw[kUnroll][NV];
#pragma unroll
        for (int uu = 0; uu < kUnroll; ++uu) {
            const int kk = base + uu * kKeysPerRound + warp * KPW + half;
#pragma unroll
            for (int i = 0; i < NV; ++i) raw[uu][i] = make_uint4(0u, 0u, 0u, 0u);
            if (kk < nk) {
                const uint16_t *r = row_ptr<D, DL>(a, a.v, s, g, k0 + kk, sub, err);
                if (r) load_slice<DL>(r, raw[uu]);
            }
        }
#pragma unroll
        for (int uu = 0; uu < kUnroll; ++uu) {
            const int kk = base + uu * kKeysPerRound + warp * KPW + half;
            if (kk < nk) {
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    float vf[8];
                    bf16x8_to_f32(raw[uu][i], vf);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float p = logit[h][kk];
#pragma unroll
                        for (int e = 0; e < E; ++e) acc[h][8 * i + e] = fmaf(p, vf[e], acc[h][8 * i + e]);
                    }
                }
            }
        }
    }
    // the two key slots of a warp, then the 8 warps, in a fixed order
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < DL; ++e)
#pragma unroll
            for (int o = kLanesPerKey; o < 32; o <<= 1) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], o);
    if (half == 0)
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < DL; ++e) red[warp][h][sub * DL + e] = acc[h][e];
    __syncthreads();
    for (int i = threadIdx.x; i < G * D; i += kDecThreads) {
        const int h = i / D, d = i % D;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kDecThreads / 32; ++w) v += red[w][h][d];
        const int64_t idx = ((int64_t)s * a.hq + g * G + h) * a.max_splits + sp;
        a.part[idx * D + d] = v;
        if (d == 0) a.stat[idx] = st_m[h];
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
    const size_t smem = sizeof(float) * ((size_t)G * kSplit + (size_t)(kDecThreads / 32) * G * D);
    auto kern = decode_split_kernel<D, G>;
    if (smem > 47 * 1024) {  // with the static part, above the default 48 KB
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
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
    const dim3 grid((unsigned)a.max_splits, (unsigned)a.hkv, (unsigned)n);
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
