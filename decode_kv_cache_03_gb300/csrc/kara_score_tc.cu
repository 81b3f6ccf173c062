// Window scoring on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Follows the gist.science summary of Kara (arXiv 2607.01237), section
// "1. Sliding-Window Bidirectional Attention Scoring" (Mechanism, Rationale):
// the query states of all W window tokens score the keys of the window with
// bidirectional attention (no causal mask) and the attention weights are
// accumulated.  For window u = (sequence, layer, KV head g):
//     p[h,i,j] = softmax_j( <q_{h,i}, k_j> / sqrt(D) ),  i, j < W, h in group g
//     s[j]     = sum_h sum_i p[h,i,j],  j < C = W - B
// The softmax of a query row runs over all W window keys; keys j >= C (the
// protected buffer) take part in the normalisation but are not scored.
//
// Work decomposition: one thread-block cluster per window, one CTA per slice of
// up to 256 window keys (cluster size ceil(W/256) <= 8).  Each CTA gathers its
// key slice once through the block table into shared memory (128-byte
// swizzled, the layout the tensor core reads) and streams the window's query
// rows through a TMA ring of 128-row strips, twice:
//
//   pass 1  S = Q_strip * K_slice^T  (M = 128 query rows, N = slice) into TMEM;
//           each half of the softmax warps takes half of the slice's keys
//           and keeps, per row, the log2 of its sum of 2^l2 (fp32, shifted
//           by its maximum); the cluster then merges these 2*ncta partials
//           through distributed shared memory into
//           lse2[row] = log2 sum_j 2^(l2_j), l2 = <q,k> * log2(e)/sqrt(D).
//   pass 2  S^T = K_tile * Q_strip^T (M = 128 keys of the slice's compressible
//           part, N = 128 query rows): key rows sit on TMEM lanes, so each
//           thread owns one key and sums 2^(l2 - lse2[row]) over its row of
//           TMEM -- the column sum needs no cross-thread reduction.
//
// No W x W matrix ever reaches memory; every score is a deterministic fp32 sum.
//
// Warp roles (320 threads): warp 0 issues TMA loads, warp 1 allocates TMEM and
// issues MMAs (one elected lane), warps 2..9 read TMEM (softmax / sums).  Every
// wait on an mbarrier is bounded; on time-out the CTA records KARA_ETIMEOUT,
// stops issuing work, drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "kara_common.cuh"
#include "kara_sm100.cuh"

namespace kara {
namespace {

using namespace ptx;

constexpr int kSlice = 256;        // keys per CTA
constexpr int kStrip = 128;        // query rows per strip
constexpr int kMaxStages = 4;
constexpr int kMaxGW = 8192;       // query rows per window (G*W) the kernel supports

// Warp roles: warp 0 issues TMA, warp 1 issues MMAs, then 4*NG softmax warps in
// NG column groups (four warps per group cover the 128 TMEM lanes).
template <int NG>
struct Roles {
    static constexpr int kSoft = 128 * NG;        // softmax threads
    static constexpr int kThreads = 64 + kSoft;
    static constexpr int kRows = kMaxGW / kSoft;  // query rows per softmax thread, at most
};
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s: every wait here normally ends in microseconds

template <int D>
struct Cfg {
    static constexpr int kAtoms = D / 64;              // 128-byte swizzle atoms per row
    static constexpr int kKBytes = kSlice * D * 2;
    static constexpr int kQBytes = kStrip * D * 2;
    static constexpr int kKAtomBytes = kSlice * 128;   // one atom of the key slice
    static constexpr int kQAtomBytes = kStrip * 128;   // one atom of a query strip
    static constexpr int kKSteps = D / 16;
};

struct Shared {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    int bad;
    uint64_t wait_ns;               // limit of the waits on progress (debug_stall)
    int32_t sblk[kSlice / 16 + 2];  // block ids of this CTA's key slice (16-token blocks)
};

// Dynamic shared memory of one CTA.  Never below 120 KB: with more than half
// of the SM's shared memory no second CTA can share the SM, so a CTA never
// waits in tcgen05.alloc for TMEM that a cluster peer on the same SM holds
// while that peer waits for it at a cluster barrier.
constexpr size_t kMinSmem = 120 * 1024;

size_t smem_bytes(int D, int T, int stages, int NG)
{
    const size_t kb = (size_t)kSlice * D * 2, qb = (size_t)kStrip * D * 2;
    const size_t need = 1024 + kb + stages * qb + (size_t)T * kStrip * 4 * NG + sizeof(Shared);
    return need > kMinSmem ? need : kMinSmem;
}

// Bounded wait on an mbarrier phase.  Returns false (without waiting) once the
// CTA has aborted, or after recording a time-out.
__device__ bool wait_phase(uint32_t bar, uint32_t parity, Shared *sh, int32_t *err, bool honour_abort = true)
{
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u) {
            if (honour_abort && *(volatile int *)&sh->abort) return false;
            const uint64_t now = globaltimer();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > (honour_abort ? sh->wait_ns : kTimeoutNs)) {
                set_err(err, KARA_ETIMEOUT);
                *(volatile int *)&sh->abort = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ float fv(uint32_t x) { return __uint_as_float(x); }

// Max of 32 fp32 values (raw bits), a tree of 3-input max of depth 4.
__device__ __forceinline__ float max32(const uint32_t (&v)[32])
{
    float a[11];
#pragma unroll
    for (int i = 0; i < 10; ++i) a[i] = max3(fv(v[3 * i]), fv(v[3 * i + 1]), fv(v[3 * i + 2]));
    a[10] = fmaxf(fv(v[30]), fv(v[31]));
    const float b0 = max3(a[0], a[1], a[2]), b1 = max3(a[3], a[4], a[5]), b2 = max3(a[6], a[7], a[8]);
    return max3(max3(b0, b1, b2), a[9], a[10]);
}

// 2^y for a pair of values on the special-function unit.  (Sending a share of
// the pairs to the FMA-pipe polynomial exp2_poly2 was measured slower here:
// the exponential unit is not what bounds this kernel.)
template <int SLOT>
__device__ __forceinline__ uint64_t exp2_pair(uint64_t y)
{
    float y0, y1;
    unpack2(y, y0, y1);
    return pack2(ex2(y0), ex2(y1));
}

// acc[j] += 2^(x*c2 + nm) for 32 values, as 4 packed pairs of partial sums.
__device__ __forceinline__ void exp_sum32(const uint32_t (&v)[32], uint64_t c2p, uint64_t nmp, uint64_t (&acc)[4])
{
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        const uint64_t y0 = fma2(pack2(fv(v[i + 0]), fv(v[i + 1])), c2p, nmp);
        const uint64_t y1 = fma2(pack2(fv(v[i + 2]), fv(v[i + 3])), c2p, nmp);
        const uint64_t y2 = fma2(pack2(fv(v[i + 4]), fv(v[i + 5])), c2p, nmp);
        const uint64_t y3 = fma2(pack2(fv(v[i + 6]), fv(v[i + 7])), c2p, nmp);
        acc[0] = add2(acc[0], exp2_pair<0>(y0));
        acc[1] = add2(acc[1], exp2_pair<1>(y1));
        acc[2] = add2(acc[2], exp2_pair<2>(y2));
        acc[3] = add2(acc[3], exp2_pair<3>(y3));
    }
}

// acc[j] += 2^(x_n*c2 + nl[n]) for the 32 columns n of one TMEM load; nl is 16-byte aligned.
__device__ __forceinline__ void exp_sum32_cols(const uint32_t (&v)[32], uint64_t c2p, const float *nl,
                                               uint64_t (&acc)[4])
{
    const float4 *n4 = reinterpret_cast<const float4 *>(nl);
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        const float4 qa = n4[i >> 2], qb = n4[(i >> 2) + 1];
        const uint64_t y0 = fma2(pack2(fv(v[i + 0]), fv(v[i + 1])), c2p, pack2(qa.x, qa.y));
        const uint64_t y1 = fma2(pack2(fv(v[i + 2]), fv(v[i + 3])), c2p, pack2(qa.z, qa.w));
        const uint64_t y2 = fma2(pack2(fv(v[i + 4]), fv(v[i + 5])), c2p, pack2(qb.x, qb.y));
        const uint64_t y3 = fma2(pack2(fv(v[i + 6]), fv(v[i + 7])), c2p, pack2(qb.z, qb.w));
        acc[0] = add2(acc[0], exp2_pair<0>(y0));
        acc[1] = add2(acc[1], exp2_pair<1>(y1));
        acc[2] = add2(acc[2], exp2_pair<2>(y2));
        acc[3] = add2(acc[3], exp2_pair<3>(y3));
    }
}

__device__ __forceinline__ float sum_pairs(const uint64_t (&acc)[4])
{
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float lo, hi;
        unpack2(acc[j], lo, hi);
        s += lo + hi;
    }
    return s;
}

// Merges the NG per-column-group log2-sum-exp values of query rows r0,
// r0 + kSoft, ... below r_hi over the cluster's ncta slices and stores
// -lse2 = -log2 sum 2^(l - max) - max into the first value of the row in
// every CTA.  NR rows at a time, all NR * ncta remote loads in flight before
// any is used.
template <int NR, int NP, int NG>
__device__ __forceinline__ void merge_rows(uint32_t part_u32, int r0, int r_hi, int ncta)
{
    constexpr int kSoft = Roles<NG>::kSoft;
    for (; r0 < r_hi; r0 += NR * kSoft) {
        float pr[NR][NP][NG];
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            const int r = r0 + k * kSoft;
#pragma unroll
            for (int cr = 0; cr < NP; ++cr)
                if (r < r_hi && cr < ncta) {
                    static_assert(NG == 2, "two partials per row");
                    const float2 x = ld_cluster_f2(mapa(part_u32 + 4u * NG * r, (uint32_t)cr));
                    pr[k][cr][0] = x.x, pr[k][cr][1] = x.y;
                }
        }
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            const int r = r0 + k * kSoft;
            if (r >= r_hi) continue;
            float M = -INFINITY;
#pragma unroll
            for (int cr = 0; cr < NP; ++cr)
                if (cr < ncta)
#pragma unroll
                    for (int q = 0; q < NG; ++q) M = fmaxf(M, pr[k][cr][q]);
            float Z = 0.f;
#pragma unroll
            for (int cr = 0; cr < NP; ++cr)
                if (cr < ncta)
#pragma unroll
                    for (int q = 0; q < NG; ++q) Z += ex2(pr[k][cr][q] - M);
            const float nl = -(M + log2f(Z));
#pragma unroll
            for (int cr = 0; cr < NP; ++cr)
                if (cr < ncta) st_cluster_f32(mapa(part_u32 + 4u * NG * r, (uint32_t)cr), nl);
        }
    }
}

// Pass 1 of one softmax thread (query row `row` of every strip, the
// NLD * 32 keys of its column group cg): for each strip, waits for the S tile
// in TMEM buffer t & 1, releases the buffer once its columns are in
// registers, and stores log2 sum 2^l2 over those keys (shifted by their
// maximum) at lse_part[NG * r + cg].  NLD is a template parameter so that one
// strip's loads, maxima and exponentials form a single branch-free block.
template <int NLD, bool CAUSAL, int NG>
__device__ __forceinline__ void pass1_rows(Shared *sh, int32_t *err, uint32_t ta0, int row, int cg, int T, int GW,
                                           float c2, float *lse_part, int W, int key0)
{
    const int lane = threadIdx.x & 31;
    for (int t = 0; t < T; ++t) {
        const int b = t & 1;
        wait_phase(smem_u32(&sh->tfull[b]), (t >> 1) & 1, sh, err);
        tc_fence_after();
        uint32_t v[NLD][32];
#pragma unroll
        for (int k = 0; k < NLD; ++k) tmem_ld32(ta0 + b * 256 + k * 32, v[k]);
#pragma unroll
        for (int k = 0; k < NLD; ++k) tmem_wait_ld(v[k]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[b]));
        if (CAUSAL) {
            // query i = r mod W sees keys key0 + col <= i only: later columns become -inf
            const int lim = (t * kStrip + row) % W - key0;
            if (!__all_sync(0xffffffffu, lim >= NLD * 32 - 1)) {
#pragma unroll
                for (int k = 0; k < NLD; ++k)
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (k * 32 + c > lim) v[k][c] = 0xff800000u;
            }
        }
        float m = max32(v[0]);
#pragma unroll
        for (int k = 1; k < NLD; ++k) m = fmaxf(m, max32(v[k]));
        // (causal) a row whose keys here are all masked gives z = 0 and lse -inf
        const float mc = (CAUSAL && m == -INFINITY) ? 0.f : m * c2;
        uint64_t acc[4] = {0, 0, 0, 0};
        const uint64_t c2p = pack2(c2, c2), nmp = pack2(-mc, -mc);
#pragma unroll
        for (int k = 0; k < NLD; ++k) exp_sum32(v[k], c2p, nmp, acc);
        const float z = sum_pairs(acc);
        // z >= 1, as the maximum contributes 2^0.  The column groups of a row
        // stay separate until the cluster merge, so no warp waits for another.
        const int r = t * kStrip + row;
        if (r < GW) lse_part[NG * r + cg] = mc + log2f(z);
    }
}

// CAUSAL: the scoring ablation without bidirectional attention (query i sees
// keys j <= i); a template parameter so that the default path carries no mask code.
// NG: column groups of softmax warps (Roles).
template <int D, bool CAUSAL, int NG>
__global__ void __launch_bounds__(Roles<NG>::kThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmap, const Geo g, float *__restrict__ scores,
                    int32_t *err, int ncta, int T, int stages, float c2, uint64_t wait_ns, int stall)
{
    using C_ = Cfg<D>;
    constexpr int kSoft = Roles<NG>::kSoft, kThreads = Roles<NG>::kThreads, kRows = Roles<NG>::kRows;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *sK = base;
    uint8_t *sQ = sK + C_::kKBytes;
    float *part = reinterpret_cast<float *>(sQ + stages * C_::kQBytes);  // per row: NG partial lse2
    Shared *sh = reinterpret_cast<Shared *>(part + T * kStrip * NG);
    const uint32_t sK_u = smem_u32(sK), sQ_u = smem_u32(sQ);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const int64_t u = blockIdx.x / ncta;
    int s, l, h;
    window_coords(g, u, s, l, h);
    const int GW = g.G * g.W;
    const int slice0 = (int)crank * kSlice;
    const int S = min(kSlice, g.W - slice0);                // keys of this CTA (multiple of 64)
    const int Cc = max(0, min(S, g.C - slice0));            // compressible keys of this CTA
    const int nM = (Cc + 127) / 128;                        // pass-2 M tiles (0..2)
    const int T2 = nM > 0 ? T : 0;

    // -- validity of the window (uniform over the cluster) --------------------
    const int32_t L = g.len[s];
    bool valid = L >= g.W && ((int64_t)L + g.bs - 1) / g.bs <= g.bt_stride;
    if (threadIdx.x == 0) { sh->abort = 0; sh->bad = 0; sh->wait_ns = wait_ns; }
    __syncthreads();
    const int32_t ws = L - g.W;
    const int32_t *btr = g.bt + (int64_t)s * g.bt_stride;
    // every block of the window is checked; the slice's own ids are kept in
    // shared memory, so the gather below issues its copies without waiting on
    // table loads
    const int fb = (ws + slice0) / g.bs;  // first logical block of the slice
    if (valid) {
        const int nb = (L + g.bs - 1) / g.bs - ws / g.bs;
        const int nbs = (ws + slice0 + S - 1) / g.bs - fb + 1;
        for (int t = threadIdx.x; t < nb; t += kThreads) {
            const int lb = ws / g.bs + t;
            const int32_t b = btr[lb];
            if (b < 0 || b >= g.num_blocks) sh->bad = 1;
            if (lb >= fb && lb < fb + nbs) sh->sblk[lb - fb] = b;
        }
    }
    __syncthreads();
    if (!valid || sh->bad) {
        if (threadIdx.x == 0) set_err(err, valid ? KARA_EBADBLOCK : KARA_EINVAL);
        for (int j = threadIdx.x; j < Cc; j += kThreads) scores[u * g.C + slice0 + j] = 0.f;
        return;
    }

    // -- set-up: barriers, TMEM, key slice -------------------------------------
    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(smem_u32(&sh->full[i]), 1);
            mbar_init(smem_u32(&sh->empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sh->tfull[i]), 1);
            mbar_init(smem_u32(&sh->tempty[i]), kSoft / 32);
        }
        mbar_init(smem_u32(&sh->done), 1);
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sh->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) prefetch_tmap(&tmap);
    // Key rows slice0 .. slice0+S-1 of the window, 16 bytes per copy, written in
    // the 128-byte swizzled K-major layout: chunk c of row r of atom a lands at
    // atom_base + r*128 + ((c ^ (r & 7)) * 16).
    {
        constexpr int CPR = D / 8;  // 16-byte chunks per row
        for (int idx = threadIdx.x; idx < S * CPR; idx += kThreads) {
            const int r = idx / CPR, cc = idx % CPR;
            const int x = ws + slice0 + r;
            const int32_t blk = sh->sblk[x / g.bs - fb];
            const uint16_t *src = g.k + pool_off(g, l, blk, h, x % g.bs) + cc * 8;
            const int a = cc >> 3, c8 = cc & 7;
            const uint32_t dst = sK_u + a * C_::kKAtomBytes + r * 128 + ((c8 ^ (r & 7)) << 4);
            cp_async16(dst, src);
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;

    if (warp == 0) {
        // ---------------- producer: query strips by TMA ----------------------
        const int row0 = ((s * g.layers + l) * g.hq + h * g.G) * g.W;
        const int pre = min(stages, T2);
        int issued = 0;
        auto produce = [&](int j) {
            const int st = j % stages;
            if (!wait_phase(smem_u32(&sh->empty[st]), ((j / stages) & 1) ^ 1, sh, err)) return;
            const uint32_t fb = smem_u32(&sh->full[st]);
            mbar_arrive_expect_tx(fb, C_::kQBytes);
            const int t = j < T ? j : j - T;
#pragma unroll
            for (int a = 0; a < C_::kAtoms; ++a)
                tma_load_2d(sQ_u + st * C_::kQBytes + a * C_::kQAtomBytes, &tmap, fb, a * 64, row0 + t * kStrip);
            issued = j + 1;
        };
        if (lane == 0 && !stall)
            for (int j = 0; j < T + pre; ++j) produce(j);
        __syncwarp();
        cluster_arrive();
        cluster_wait();
        cluster_arrive();
        if (lane == 0) {
            if (!stall)
                for (int j = T + pre; j < T + T2; ++j) produce(j);
            // drain: every issued copy has landed before this CTA may exit
            for (int j = max(0, issued - stages); j < issued; ++j)
                wait_phase(smem_u32(&sh->full[j % stages]), (j / stages) & 1, sh, err, false);
        }
        __syncwarp();
        cluster_wait();
    } else if (warp == 1) {
        // ---------------- MMA issuer -----------------------------------------
        const uint32_t idesc1 = idesc_bf16(128, S);
        const uint32_t idesc2 = idesc_bf16(128, 128);
        if (lane == 0) {
            for (int t = 0; t < T; ++t) {
                const int st = t % stages, b = t & 1;
                if (!wait_phase(smem_u32(&sh->full[st]), (t / stages) & 1, sh, err)) break;
                if (!wait_phase(smem_u32(&sh->tempty[b]), ((t >> 1) & 1) ^ 1, sh, err)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C_::kKSteps; ++kk) {
                    const int a = kk >> 2, off = (kk & 3) * 32;
                    const uint64_t ad = sdesc_sw128(sQ_u + st * C_::kQBytes + a * C_::kQAtomBytes + off);
                    const uint64_t bd = sdesc_sw128(sK_u + a * C_::kKAtomBytes + off);
                    mma_bf16(tmem + b * 256, ad, bd, idesc1, kk > 0);
                }
                mma_commit(smem_u32(&sh->empty[st]));
                mma_commit(smem_u32(&sh->tfull[b]));
            }
        }
        __syncwarp();
        cluster_arrive();
        cluster_wait();
        cluster_arrive();
        if (lane == 0) {
            for (int t = 0; t < T2; ++t) {
                const int j = T + t, st = j % stages, b = j & 1;
                if (!wait_phase(smem_u32(&sh->full[st]), (j / stages) & 1, sh, err)) break;
                if (!wait_phase(smem_u32(&sh->tempty[b]), ((j >> 1) & 1) ^ 1, sh, err)) break;
                tc_fence_after();
                for (int mt = 0; mt < nM; ++mt) {
#pragma unroll
                    for (int kk = 0; kk < C_::kKSteps; ++kk) {
                        const int a = kk >> 2, off = (kk & 3) * 32;
                        const uint64_t ad = sdesc_sw128(sK_u + a * C_::kKAtomBytes + mt * (128 * 128) + off);
                        const uint64_t bd = sdesc_sw128(sQ_u + st * C_::kQBytes + a * C_::kQAtomBytes + off);
                        mma_bf16(tmem + b * 256 + mt * 128, ad, bd, idesc2, kk > 0);
                    }
                }
                mma_commit(smem_u32(&sh->empty[st]));
                mma_commit(smem_u32(&sh->tfull[b]));
            }
            // every MMA issued has completed before TMEM is freed
            mma_commit(smem_u32(&sh->done));
            wait_phase(smem_u32(&sh->done), 0, sh, err, false);
        }
        __syncwarp();
        cluster_wait();
    } else {
        // ---------------- softmax / column sums (warps 2 ..) ---------------------
        const int sw = warp - 2, q4 = warp & 3, cg = sw >> 2;  // TMEM lane quarter, column group
        const int row = 32 * q4 + lane;
        const int sidx = sw * 32 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const int cols = S / NG;   // pass-1 keys of this column group
        const int nld = cols >> 5; // 32-column loads: 1..4

        // pass 1: per row, log2-sum-exp over this column group's keys of the slice
        const uint32_t ta1 = tmem + lane_base + cg * cols;
        const int key0 = slice0 + cg * cols;
        if (nld == 1) {
            pass1_rows<1, CAUSAL, NG>(sh, err, ta1, row, cg, T, GW, c2, part, g.W, key0);
        } else if (nld == 2) {
            pass1_rows<2, CAUSAL, NG>(sh, err, ta1, row, cg, T, GW, c2, part, g.W, key0);
        } else if (nld == 3) {
            pass1_rows<3, CAUSAL, NG>(sh, err, ta1, row, cg, T, GW, c2, part, g.W, key0);
        } else {
            pass1_rows<4, CAUSAL, NG>(sh, err, ta1, row, cg, T, GW, c2, part, g.W, key0);
        }
        __syncwarp();
        cluster_arrive();
        cluster_wait();
        // merge the column groups' lse2 of every query row: this CTA owns rows
        // [r_lo, r_hi), reads their NG values from every peer and writes -lse2
        // into the first value of the row in every peer
        const int TT = T * kStrip;
        {
            const int P = (GW + ncta - 1) / ncta;
            const int r_lo = min(GW, (int)crank * P), r_hi = min(GW, r_lo + P);
            const uint32_t pa = smem_u32(part);
            // NR * NP * NG = 64 values in flight per thread
            if (ncta <= 4)
                merge_rows<16 / NG, 4, NG>(pa, r_lo + sidx, r_hi, ncta);
            else
                merge_rows<8 / NG, 8, NG>(pa, r_lo + sidx, r_hi, ncta);
        }
        cluster_arrive();
        cluster_wait();
        // -lse2 of every row, packed to one float per row in place of the pairs;
        // rows past G*W (the padding of the last strip) get -inf, so they add 0
        float nlv[kRows];
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            const int r = sidx + k * kSoft;
            nlv[k] = r < GW ? part[NG * r] : -INFINITY;
        }
        named_barrier(1, kSoft);
        float *nlse2 = part;
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            const int r = sidx + k * kSoft;
            if (r < TT) nlse2[r] = nlv[k];
        }
        named_barrier(1, kSoft);

        // pass 2: column sums with keys on TMEM lanes; column group cg takes key tile cg
        constexpr int kL2 = 4;   // 32-column loads per strip
        const int mt = cg, c0 = 0;
        float acc = 0.f;
        for (int t = 0; t < T2; ++t) {
            const int j = T + t, b = j & 1;
            wait_phase(smem_u32(&sh->tfull[b]), (j >> 1) & 1, sh, err);
            tc_fence_after();
            uint32_t v[kL2][32];
            const bool mine = mt < nM;
            if (mine) {
                const uint32_t ta = tmem + lane_base + b * 256 + mt * 128 + c0;
#pragma unroll
                for (int k = 0; k < kL2; ++k) tmem_ld32(ta + k * 32, v[k]);
#pragma unroll
                for (int k = 0; k < kL2; ++k) tmem_wait_ld(v[k]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[b]));
            bool skip = false;
            if (CAUSAL && mine) {
                // key j adds the weights of queries i >= j only: column n of the
                // strip is query i = (t*128 + n) mod W
                const int jk = slice0 + mt * 128 + row, i0 = (t * kStrip) % g.W;
                const bool wraps = i0 + kStrip > g.W;
                const bool all_in = !wraps && i0 >= jk;
                const bool all_out = !wraps && i0 + kStrip - 1 < jk;
                skip = __all_sync(0xffffffffu, all_out);
                if (!skip && !__all_sync(0xffffffffu, all_in)) {
#pragma unroll
                    for (int k = 0; k < kL2; ++k)
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            int i = i0 + c0 + k * 32 + c;
                            if (i >= g.W) i -= g.W;
                            if (i < jk) v[k][c] = 0xff800000u;
                        }
                }
            }
            if (mine && !skip) {
                const float *nl = nlse2 + t * kStrip + c0;
                uint64_t pacc[4] = {0, 0, 0, 0};
                const uint64_t c2p = pack2(c2, c2);
#pragma unroll
                for (int k = 0; k < kL2; ++k) exp_sum32_cols(v[k], c2p, nl + k * 32, pacc);
                acc += sum_pairs(pacc);
            }
        }
        const int key = slice0 + mt * 128 + row;
        if (mt < nM && key < g.C) scores[u * g.C + key] = acc;
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

namespace {

template <int D>
cudaError_t launch_tc(const Geo &g, float *scores, int32_t *err, cudaStream_t st)
{
    const int ncta = (g.W + kSlice - 1) / kSlice;
    const int T = (g.G * g.W + kStrip - 1) / kStrip;
    // Two column groups of softmax warps.  Four (16 softmax warps) made pass 1
    // 7 % faster but pass 2 13 % slower on the Qwen3-14B shape: with four busy
    // softmax warps per SM sub-partition, the MMA-issuing warp falls behind.
    constexpr int NG = 2;
    int stages = kMaxStages;
    while (stages > 2 && smem_bytes(D, T, stages, NG) > 232448) --stages;
    const size_t smem = smem_bytes(D, T, stages, NG);
    if (smem > 232448) return cudaErrorInvalidValue;

    auto fn = tensor_map_encoder();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap tmap;
    const cuuint64_t rows = (cuuint64_t)g.n * g.layers * g.hq * g.W;
    cuuint64_t dims[2] = {(cuuint64_t)D, rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kStrip};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(g.q), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

    auto kern = g.causal ? score_tc_kernel<D, true, NG> : score_tc_kernel<D, false, NG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(g.nwin * ncta));
    cfg.blockDim = dim3(Roles<NG>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ncta;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float c2 = 1.4426950408889634f / sqrtf((float)D);
    const Stall dbg = debug_stall(kTimeoutNs);
    return cudaLaunchKernelEx(&cfg, kern, tmap, g, scores, err, ncta, T, stages, c2, dbg.wait_ns, (int)dbg.on);
}

}  // namespace

size_t score_sp_scratch_bytes(const Geo &g);

// Scratch of the scoring path (the single-pass kernel's per-window marks).
size_t score_scratch_bytes(const Geo &g) { return score_sp_scratch_bytes(g); }

bool score_sp_supported(const Geo &g);
cudaError_t launch_score_sp(const Geo &g, float *scores, void *scratch, int32_t *err, cudaStream_t st);

cudaError_t launch_score(const Geo &g, float *scores, void *scratch, int32_t *err, cudaStream_t st)
{
    if (g.nwin == 0) return cudaSuccess;
    // one pass over the logits where the single-pass kernel covers the shape
    // (bidirectional, W <= 2048); the two-pass kernel for the causal ablation
    if (score_sp_supported(g)) return launch_score_sp(g, scores, scratch, err, st);
    if (g.G * g.W > 8192) return cudaErrorInvalidValue;
    return g.D == 128 ? launch_tc<128>(g, scores, err, st) : launch_tc<64>(g, scores, err, st);
}

}  // namespace kara
