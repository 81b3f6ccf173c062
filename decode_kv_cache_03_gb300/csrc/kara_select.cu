// Top-K candidates and Token2Chunk selection, one thread block per window.
//
// Follows the gist.science summary of Kara (arXiv 2607.01237): section
// "1. Sliding-Window Bidirectional Attention Scoring", Selection (the Top-K
// most important KV pairs of the window become candidates) and section
// "2. Token2Chunk Module", Process (candidates sorted by index; every two
// consecutive ones bound a chunk scored from its length and endpoint scores;
// chunks are filtered and selected).  Readings where the pages are silent:
// ties go to the lower index; the chunk score is (s_a + s_b) / (1 + lambda*len)
// in fp32 with round-to-nearest and no contraction; chunks are visited by
// (score desc, left end asc) and kept first-fit under the budget R; the budget
// is then filled to exactly R with candidates and then other positions, both
// in score order.
//
// Everything is integer or exactly-rounded fp32 work in shared memory, so the
// result is a pure function of the fp32 scores.  Top-K and the second fill use
// an MSB-first radix select on order-preserving 32-bit keys; equal keys are
// resolved by index with a block-wide prefix count.
#include "kara_common.cuh"

namespace kara {
namespace {

constexpr int kSelThreads = 256;

// Order-preserving key of a finite float; -0.0 maps to +0.0's key.
__device__ __forceinline__ uint32_t okey(float x)
{
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ int warp_incl_scan(int v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

struct SelShared {
    uint32_t hist[256];
    int scan[33];
    int digit, gt, count;
};

__device__ int block_excl_scan(int v, SelShared &sh, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int nw = kSelThreads / 32;
    int incl = warp_incl_scan(v);
    if (lane == 31) sh.scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = lane < nw ? sh.scan[lane] : 0;
        int xi = warp_incl_scan(x);
        if (lane < nw) sh.scan[lane] = xi - x;
        if (lane == 31) sh.scan[32] = xi;
    }
    __syncthreads();
    const int r = sh.scan[warp] + incl - v;
    *total = sh.scan[32];
    __syncthreads();
    return r;
}

// Marks in `flag` the `need` eligible positions that come first in the order
// (score desc, index asc).  Requires need <= number of eligible positions.
// Each thread owns the contiguous index range [lo, hi).
template <class Elig>
__device__ void radix_take(const float *s, int lo, int hi, int need, Elig elig, uint8_t *flag,
                           SelShared &sh)
{
    uint32_t prefix = 0u, pmask = 0u;
    int remaining = need;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kSelThreads) sh.hist[i] = 0u;
        __syncthreads();
        for (int j = lo; j < hi; ++j) {
            if (!elig(j)) continue;
            const uint32_t k = okey(s[j]);
            if ((k & pmask) == prefix) atomicAdd(&sh.hist[(k >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            int cnt[8];
            int tot = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                cnt[k] = (int)sh.hist[255 - 8 * lane - k];
                tot += cnt[k];
            }
            const int incl = warp_incl_scan(tot);
            const int excl = incl - tot;
            if (excl < remaining && remaining <= incl) {
                int c = excl;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (c + cnt[k] >= remaining) {
                        sh.digit = 255 - 8 * lane - k;
                        sh.gt = c;
                        break;
                    }
                    c += cnt[k];
                }
            }
        }
        __syncthreads();
        remaining -= sh.gt;
        prefix |= (uint32_t)sh.digit << shift;
        pmask |= 255u << shift;
        __syncthreads();
    }
    // prefix is the key of the need-th position; take `remaining` equal keys by index
    int neq = 0;
    for (int j = lo; j < hi; ++j)
        if (elig(j) && okey(s[j]) == prefix) ++neq;
    int tot;
    int rank = block_excl_scan(neq, sh, &tot);
    for (int j = lo; j < hi; ++j) {
        if (!elig(j)) continue;
        const uint32_t k = okey(s[j]);
        if (k > prefix) {
            flag[j] = 1;
        } else if (k == prefix) {
            if (rank < remaining) flag[j] = 1;
            ++rank;
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(int C, int K, int R, float lambda, int mode,
                                                             int chunk, const float *__restrict__ scores,
                                                             int32_t *cand_out, int32_t *kept_out)
{
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ SelShared sh;
    const int64_t u = blockIdx.x;
    const int nfc = mode == KARA_SELECT_FIXED_CHUNK ? (C + chunk - 1) / chunk : 0;  // fixed chunks
    float *s = reinterpret_cast<float *>(smem);
    int32_t *cand = reinterpret_cast<int32_t *>(s + C);
    float *cs = reinterpret_cast<float *>(cand + K);
    int32_t *corder = reinterpret_cast<int32_t *>(cs + K);
    int32_t *corder2 = corder + K;
    float *fmean = reinterpret_cast<float *>(corder2 + K);
    int32_t *forder = reinterpret_cast<int32_t *>(fmean + nfc);
    uint8_t *cflag = reinterpret_cast<uint8_t *>(forder + nfc);
    uint8_t *kflag = cflag + C;
    uint8_t *taken = kflag + C;

    const int tid = threadIdx.x;
    const int E = (C + kSelThreads - 1) / kSelThreads;
    const int lo = min(C, tid * E), hi = min(C, lo + E);
    const float *src = scores + u * C;
    for (int j = tid; j < C; j += kSelThreads) {
        s[j] = src[j];
        cflag[j] = 0;
        kflag[j] = 0;
    }
    for (int t = tid; t < K; t += kSelThreads) taken[t] = 0;
    __syncthreads();

    // 1. Top-K candidates.
    radix_take(s, lo, hi, K, [](int) { return true; }, cflag, sh);

    // 2. Candidates by index.
    int nc = 0;
    for (int j = lo; j < hi; ++j) nc += cflag[j];
    int tot;
    const int cbase = block_excl_scan(nc, sh, &tot);
    {
        int w = cbase;
        for (int j = lo; j < hi; ++j)
            if (cflag[j]) cand[w++] = j;
    }
    __syncthreads();

    if (mode == KARA_SELECT_TOP_R) {
        // Token-level Top-R: the R positions first in the score order.
        radix_take(s, lo, hi, R, [](int) { return true; }, kflag, sh);
    } else if (mode == KARA_SELECT_FIXED_CHUNK) {
        // Fixed chunks [k*chunk, min(C, (k+1)*chunk)) scored by their mean (a
        // float sum in index order, then one rounded division) ...
        for (int t = tid; t < nfc; t += kSelThreads) {
            const int a = t * chunk, b = min(C, a + chunk);
            float sum = 0.f;
            for (int j = a; j < b; ++j) sum = __fadd_rn(sum, s[j]);
            fmean[t] = __fdiv_rn(sum, (float)(b - a));
        }
        __syncthreads();
        // ... visited by (mean desc, start asc) ...
        for (int t = tid; t < nfc; t += kSelThreads) {
            const uint32_t c = okey(fmean[t]);
            int r = 0;
            for (int t2 = 0; t2 < nfc; ++t2) {
                const uint32_t c2 = okey(fmean[t2]);
                r += (c2 > c) || (c2 == c && t2 < t);
            }
            forder[r] = t;
        }
        __syncthreads();
        // ... and kept whole while they fit the budget (first fit) ...
        if (tid == 0) {
            int count = 0;
            for (int r = 0; r < nfc; ++r) {
                const int a = forder[r] * chunk, b = min(C, a + chunk);
                if (count + (b - a) <= R) {
                    for (int j = a; j < b; ++j) kflag[j] = 1;
                    count += b - a;
                }
            }
            sh.count = count;
        }
        __syncthreads();
        // ... then the budget is filled with other positions in score order.
        if (sh.count < R) {
            const int need = R - sh.count;
            __syncthreads();
            radix_take(s, lo, hi, need, [&](int j) { return !kflag[j]; }, kflag, sh);
        }
    } else {
    // 3. Chunk scores.
    const int nch = K - 1;
    for (int t = tid; t < nch; t += kSelThreads) {
        const int a = cand[t], b = cand[t + 1];
        const float num = __fadd_rn(s[a], s[b]);
        const float den = __fmaf_rn(lambda, (float)(b - a + 1), 1.0f);
        cs[t] = __fdiv_rn(num, den);
    }
    __syncthreads();

    // 4. Visit order of the chunks: (score desc, left end asc).
    for (int t = tid; t < nch; t += kSelThreads) {
        // order-preserving keys: the same order as the floats for finite
        // scores, and a total order on every bit pattern, so the ranks always
        // form a permutation (no index can go out of range on NaN input)
        const uint32_t c = okey(cs[t]);
        int r = 0;
        for (int t2 = 0; t2 < nch; ++t2) {
            const uint32_t c2 = okey(cs[t2]);
            r += (c2 > c) || (c2 == c && t2 < t);
        }
        corder[r] = t;
    }
    __syncthreads();

    // 5. First-fit greedy under the budget.  Chunk t shares its left end with
    //    chunk t-1 and its right end with chunk t+1 and nothing else.
    if (tid == 0) {
        int count = 0;
        for (int r = 0; r < nch; ++r) {
            const int t = corder[r];
            const int add = cand[t + 1] - cand[t] + 1 - (t > 0 && taken[t - 1]) -
                            (t + 1 < nch && taken[t + 1]);
            if (count + add <= R) {
                taken[t] = 1;
                count += add;
            }
        }
        sh.count = count;
    }
    __syncthreads();

    // 6. Kept flags covered by taken chunks.
    {
        int before = cbase;  // candidates with index < j
        for (int j = lo; j < hi; ++j) {
            uint8_t kf;
            if (cflag[j]) {
                const int t = before;
                kf = (t > 0 && taken[t - 1]) || (t < nch && taken[t]);
                ++before;
            } else {
                const int t = before - 1;
                kf = (t >= 0 && t < nch && taken[t]);
            }
            kflag[j] = kf;
        }
    }
    __syncthreads();

    // 7. Fill with candidates not kept yet, in score order.
    if (sh.count < R) {
        for (int t = tid; t < K; t += kSelThreads) {
            const int j = cand[t];
            const uint32_t v = okey(s[j]);
            int r = 0;
            for (int t2 = 0; t2 < K; ++t2) {
                const int j2 = cand[t2];
                const uint32_t v2 = okey(s[j2]);
                r += (v2 > v) || (v2 == v && j2 < j);
            }
            corder2[r] = t;
        }
        __syncthreads();
        if (tid == 0) {
            int count = sh.count;
            for (int r = 0; r < K && count < R; ++r) {
                const int j = cand[corder2[r]];
                if (!kflag[j]) {
                    kflag[j] = 1;
                    ++count;
                }
            }
            sh.count = count;
        }
        __syncthreads();
    }

    // 8. Fill with any other compressible position, in score order.
    if (sh.count < R) {
        const int need = R - sh.count;
        __syncthreads();
        radix_take(s, lo, hi, need, [&](int j) { return !cflag[j] && !kflag[j]; }, kflag, sh);
    }
    }  // Token2Chunk

    // 9. Outputs.
    if (cand_out)
        for (int t = tid; t < K; t += kSelThreads) cand_out[u * K + t] = cand[t];
    int nk = 0;
    for (int j = lo; j < hi; ++j) nk += kflag[j];
    const int kbase = block_excl_scan(nk, sh, &tot);
    int w = kbase;
    int32_t *ko = kept_out + u * R;
    for (int j = lo; j < hi; ++j)
        if (kflag[j] && w < R) ko[w++] = j;
}

}  // namespace

size_t select_smem_bytes(int C, int K, int mode, int chunk)
{
    const size_t nfc = mode == KARA_SELECT_FIXED_CHUNK ? (size_t)(C + chunk - 1) / chunk : 0;
    return (size_t)C * 4 + (size_t)K * 4 * 4 + nfc * 8 + (size_t)C * 2 + (size_t)K;
}

cudaError_t launch_select(int64_t nwin, int C, int K, int R, float lambda, int mode, int chunk,
                          const float *scores, int32_t *cand, int32_t *kept, cudaStream_t st)
{
    if (nwin == 0) return cudaSuccess;
    const size_t smem = select_smem_bytes(C, K, mode, chunk);
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    select_kernel<<<(unsigned)nwin, kSelThreads, smem, st>>>(C, K, R, lambda, mode, chunk, scores, cand, kept);
    return cudaGetLastError();
}

}  // namespace kara
