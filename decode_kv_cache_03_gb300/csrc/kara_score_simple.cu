// Window scoring on CUDA cores, two passes (first working path; the
// tensor-core kernel replaces it for the supported shapes).
//
// Follows the gist.science summary of Kara (arXiv 2607.01237), section
// "1. Sliding-Window Bidirectional Attention Scoring": the queries of all W
// window tokens attend, without a causal mask, to the W window keys; the
// attention weights of the compressible keys are accumulated over the window
// queries and over the query heads of the KV group.  The softmax of a query
// row runs over all W window keys and the logits are scaled by 1/sqrt(D).
//
//   pass 1 (rowstat_kernel): per query row, lse2 = log2 sum_j 2^(l2_j), with
//          l2 = <q, k> * log2(e) / sqrt(D) (online max and sum in fp32)
//   pass 2 (colsum_kernel):  per compressible key j, s[j] = sum_rows 2^(l2 - lse2)
#include <math.h>

#include "kara_common.cuh"

namespace kara {
namespace {

constexpr int kRows = 128;   // query rows (pass 1) or keys (pass 2) per block
constexpr int kTile = 32;    // keys (pass 1) or query rows (pass 2) staged per step

__device__ __forceinline__ float bf16_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Loads row `x` (logical position) of the window's K into shared memory as
// floats; returns false (and records the error) on a bad block id.
template <int D>
__device__ __forceinline__ bool window_valid(const Geo &g, int s, int32_t *err)
{
    const int32_t L = g.len[s];
    if (L < g.W || ((int64_t)L + g.bs - 1) / g.bs > g.bt_stride) {
        set_err(err, KARA_EINVAL);
        return false;
    }
    return true;
}

template <int D>
__global__ void __launch_bounds__(kRows) rowstat_kernel(Geo g, float *__restrict__ lse2, int32_t *err)
{
    __shared__ __align__(16) float kt[kTile][D];
    __shared__ int bad;
    const int64_t u = blockIdx.x;
    int s, l, h;
    window_coords(g, u, s, l, h);
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    if (!window_valid<D>(g, s, err)) return;   // uniform over the block
    const int32_t ws = g.len[s] - g.W;
    const int GW = g.G * g.W;
    const int row = blockIdx.y * kRows + threadIdx.x;
    const bool active = row < GW;
    const float c = 1.4426950408889634f * rsqrtf((float)D);

    float q[D];
    if (active) {
        const int hq = h * g.G + row / g.W, i = row % g.W;
        const uint16_t *qr = g.q + ((((int64_t)s * g.layers + l) * g.hq + hq) * g.W + i) * D;
#pragma unroll
        for (int d = 0; d < D; d += 8) {
            const uint4 v = *reinterpret_cast<const uint4 *>(qr + d);
            const uint16_t *e = reinterpret_cast<const uint16_t *>(&v);
#pragma unroll
            for (int k = 0; k < 8; ++k) q[d + k] = bf16_to_float(e[k]) * c;
        }
    }
    float m = -INFINITY, z = 0.f;
    const int32_t *btr = g.bt + (int64_t)s * g.bt_stride;
    for (int j0 = 0; j0 < g.W; j0 += kTile) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kTile * (D / 8); idx += kRows) {
            const int jj = idx / (D / 8), d = (idx % (D / 8)) * 8;
            const int x = ws + j0 + jj;
            const int32_t blk = btr[x / g.bs];
            uint4 v = make_uint4(0, 0, 0, 0);
            if (blk >= 0 && blk < g.num_blocks)
                v = *reinterpret_cast<const uint4 *>(g.k + pool_off(g, l, blk, h, x % g.bs) + d);
            else
                bad = 1;
            const uint16_t *e = reinterpret_cast<const uint16_t *>(&v);
#pragma unroll
            for (int k = 0; k < 8; ++k) kt[jj][d + k] = bf16_to_float(e[k]);
        }
        __syncthreads();
        if (active) {
#pragma unroll 4
            for (int jj = 0; jj < kTile; ++jj) {
                float acc = 0.f;
#pragma unroll
                for (int d = 0; d < D; d += 4) {
                    const float4 kv = *reinterpret_cast<const float4 *>(&kt[jj][d]);
                    acc = fmaf(q[d], kv.x, acc);
                    acc = fmaf(q[d + 1], kv.y, acc);
                    acc = fmaf(q[d + 2], kv.z, acc);
                    acc = fmaf(q[d + 3], kv.w, acc);
                }
                if (acc > m) {
                    z = z * exp2f(m - acc) + 1.f;
                    m = acc;
                } else {
                    z += exp2f(acc - m);
                }
            }
        }
    }
    __syncthreads();
    if (bad) {
        set_err(err, KARA_EBADBLOCK);
        return;
    }
    if (active) lse2[u * GW + row] = m + log2f(z);
}

template <int D>
__global__ void __launch_bounds__(kRows) colsum_kernel(Geo g, const float *__restrict__ lse2,
                                                       float *__restrict__ scores, int32_t *err)
{
    __shared__ __align__(16) float qt[kTile][D];
    __shared__ float lt[kTile];
    __shared__ int bad;
    const int64_t u = blockIdx.x;
    int s, l, h;
    window_coords(g, u, s, l, h);
    const int j = blockIdx.y * kRows + threadIdx.x;
    const bool active = j < g.C;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    if (!window_valid<D>(g, s, err)) {
        if (active) scores[u * g.C + j] = 0.f;
        return;
    }
    const int32_t ws = g.len[s] - g.W;
    const int GW = g.G * g.W;
    const float c = 1.4426950408889634f * rsqrtf((float)D);
    const int32_t *btr = g.bt + (int64_t)s * g.bt_stride;
    // every block id of the window is checked so a bad one zeroes the window
    for (int x = ws + threadIdx.x * g.bs; x < ws + g.W + g.bs; x += kRows * g.bs) {
        const int xx = min(x, ws + g.W - 1);
        const int32_t blk = btr[xx / g.bs];
        if (blk < 0 || blk >= g.num_blocks) bad = 1;
    }
    float kr[D];
    if (active) {
        const int x = ws + j;
        const int32_t blk = btr[x / g.bs];
        if (blk >= 0 && blk < g.num_blocks) {
            const uint16_t *kp = g.k + pool_off(g, l, blk, h, x % g.bs);
#pragma unroll
            for (int d = 0; d < D; d += 8) {
                const uint4 v = *reinterpret_cast<const uint4 *>(kp + d);
                const uint16_t *e = reinterpret_cast<const uint16_t *>(&v);
#pragma unroll
                for (int k = 0; k < 8; ++k) kr[d + k] = bf16_to_float(e[k]) * c;
            }
        } else {
#pragma unroll
            for (int d = 0; d < D; ++d) kr[d] = 0.f;
        }
    }
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) set_err(err, KARA_EBADBLOCK);
        if (active) scores[u * g.C + j] = 0.f;
        return;
    }
    float acc = 0.f;
    const uint16_t *qbase = g.q + (((int64_t)s * g.layers + l) * g.hq + (int64_t)h * g.G) * g.W * D;
    for (int r0 = 0; r0 < GW; r0 += kTile) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kTile * (D / 8); idx += kRows) {
            const int rr = idx / (D / 8), d = (idx % (D / 8)) * 8;
            const uint4 v = *reinterpret_cast<const uint4 *>(qbase + (int64_t)(r0 + rr) * D + d);
            const uint16_t *e = reinterpret_cast<const uint16_t *>(&v);
#pragma unroll
            for (int k = 0; k < 8; ++k) qt[rr][d + k] = bf16_to_float(e[k]);
        }
        if (threadIdx.x < kTile) lt[threadIdx.x] = lse2[u * GW + r0 + threadIdx.x];
        __syncthreads();
        if (active) {
#pragma unroll 4
            for (int rr = 0; rr < kTile; ++rr) {
                float dot = 0.f;
#pragma unroll
                for (int d = 0; d < D; d += 4) {
                    const float4 qv = *reinterpret_cast<const float4 *>(&qt[rr][d]);
                    dot = fmaf(kr[d], qv.x, dot);
                    dot = fmaf(kr[d + 1], qv.y, dot);
                    dot = fmaf(kr[d + 2], qv.z, dot);
                    dot = fmaf(kr[d + 3], qv.w, dot);
                }
                acc += exp2f(dot - lt[rr]);
            }
        }
    }
    if (active) scores[u * g.C + j] = acc;
}

}  // namespace

size_t score_scratch_bytes(const Geo &g) { return align256((size_t)g.nwin * g.G * g.W * sizeof(float)); }

cudaError_t launch_score(const Geo &g, float *scores, void *scratch, int32_t *err, cudaStream_t st)
{
    if (g.nwin == 0) return cudaSuccess;
    float *lse2 = static_cast<float *>(scratch);
    const dim3 g1((unsigned)g.nwin, (g.G * g.W + kRows - 1) / kRows);
    const dim3 g2((unsigned)g.nwin, (g.C + kRows - 1) / kRows);
    if (g.D == 128) {
        rowstat_kernel<128><<<g1, kRows, 0, st>>>(g, lse2, err);
        colsum_kernel<128><<<g2, kRows, 0, st>>>(g, lse2, scores, err);
    } else {
        rowstat_kernel<64><<<g1, kRows, 0, st>>>(g, lse2, err);
        colsum_kernel<64><<<g2, kRows, 0, st>>>(g, lse2, scores, err);
    }
    return cudaGetLastError();
}

}  // namespace kara
