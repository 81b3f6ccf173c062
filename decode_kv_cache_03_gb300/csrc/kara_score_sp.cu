// Window scoring in a single pass over the logits (tcgen05 + TMEM + TMA + DSMEM).
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
// Each logit is computed and exponentiated exactly once:
//
//   * One thread-block cluster per window, one CTA per slice of <= 256 window
//     keys (cluster size ceil(W/256) <= 4).  The key slice comes into shared
//     memory by TMA, one 16-row paged block at a time through a 5-D tensor map
//     over the pool (128-byte swizzled, the tensor core's K-major layout); the
//     window's first key may sit o rows into its block, so the MMA operand
//     starts o rows into the buffer.  The G*W query rows of the window stream
//     through a TMA ring in 128-row strips.
//   * Per strip, S = Q_strip * K_slice^T (M = 128 rows, N = slice) goes into
//     one of two TMEM buffers.  Each softmax thread owns one query row (TMEM
//     lane) and half of the slice's keys.  It exponentiates its logits once,
//     e = 2^(l2 - r) with l2 = <q,k> log2(e)/sqrt(D) and r a reference at or
//     above their maximum, and writes e back over S in TMEM.  The two halves of
//     a row merge their (r, sum e) in shared memory and one thread sends the
//     CTA's partial to every CTA of the cluster with st.async (DSMEM,
//     completing bytes on the receiver's mbarrier).
//   * When the ncta partials of its row have arrived, the thread knows the
//     row's normaliser Z = sum_c z_c 2^(r_c - M) exactly, reads e back from
//     TMEM and accumulates e * 2^(r - M) / Z into registers, one accumulator
//     per (row lane, key).  That releases the TMEM buffer for the next strip.
//   * After the window's last strip the accumulators are summed across the 32
//     lanes of each warp (a butterfly that leaves each lane whole keys) and
//     across the four lane quarters through shared memory, in a fixed order.
//
// The kernel is persistent: each cluster walks its share of the windows, and
// the next window's key slice loads into the second key buffer while the
// current window is scored.  No W x W matrix and no per-row statistic reaches
// global memory; every score is a deterministic fp32 sum.  Warp roles (384
// threads): warp 0 issues TMA loads, warp 1 allocates TMEM and issues MMAs (one
// lane), warps 2..3 idle, warps 4..11 are the softmax warps; the first
// warpgroup hands most of its registers to the softmax warpgroups.  Every wait
// is bounded; on time-out the CTA records KARA_ETIMEOUT and stops waiting,
// still draining what it has in flight.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "kara_common.cuh"
#include "kara_sm100.cuh"

namespace kara {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace {

using namespace ptx;

constexpr int kSlice = 256;    // keys per CTA
constexpr int kStrip = 128;    // query rows per strip
constexpr int kMaxCta = 4;     // CTAs per cluster: W <= 1024
constexpr int kSlots = 3;      // exchange slots (strips in flight between CTAs)
constexpr int kSoft = 256;     // softmax threads: two per TMEM lane
constexpr int kThreads = 128 + kSoft;  // three warpgroups: producer/MMA, two of softmax
// Registers per thread: at launch (65536 / 384, what ptxas assigns under the
// launch bounds), then after the warpgroups trade registers.  The trade must
// add up: 128 * kRegsLow + 256 * kRegsHigh == 384 * kRegsLaunch.
constexpr int kRegsLaunch = 168;
constexpr uint32_t kRegsLow = 40;
constexpr uint32_t kRegsHigh = 232;
static_assert(128 * kRegsLow + 256 * kRegsHigh == 384 * kRegsLaunch, "register trade must add up");
constexpr uint32_t kTmemCols = 512;
constexpr float kMargin = 8.f;  // log2 headroom of the reference above a chunk's maximum
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr int kBlockRows = 16;                         // rows of a paged block
constexpr int kSliceBlocks = kSlice / kBlockRows + 1;  // blocks a slice can touch (17)
constexpr int kKAtomBytes = kSliceBlocks * kBlockRows * 128;  // one 64-column atom of a key buffer

template <int D>
struct Cfg {
    static constexpr int kAtoms = D / 64;             // 128-byte swizzle atoms per row
    static constexpr int kKBytes = kAtoms * kKAtomBytes;
    static constexpr int kQBytes = kStrip * D * 2;
    static constexpr int kQAtomBytes = kStrip * 128;
    static constexpr int kKSteps = D / 16;
    static constexpr int kBoxBytes = kBlockRows * 128;  // one (block, atom) TMA box
};

struct Shared {
    uint64_t qfull[2], qempty[2];    // query-strip stages
    uint64_t kfull[2], kempty[2];    // key-slice buffers
    uint64_t tfull[2], tempty[2];    // TMEM buffers
    uint64_t xfull[kSlots];          // exchange slots
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    uint64_t wait_ns;
    int wbad[2];                     // 1 + index of the last window (by parity) with a bad block id
};

// Exchange slot: the partial (reference, sum) of every CTA for each row.
constexpr int kSlotFloats2 = kMaxCta * kStrip;

template <int D>
size_t smem_bytes()
{
    using C_ = Cfg<D>;
    const size_t need = 1024 + 2 * (size_t)C_::kKBytes + 2 * (size_t)C_::kQBytes
                      + (size_t)kSlots * kSlotFloats2 * 8 + 2 * kStrip * 8 + 4 * kSlice * 4 + sizeof(Shared);
    // more than half of the SM's shared memory: a second CTA never shares the
    // SM and waits in tcgen05.alloc for the TMEM this persistent one holds
    const size_t floor_ = 120 * 1024;
    return need > floor_ ? need : floor_;
}

// Bounded wait on an mbarrier phase.  Returns false (without waiting) once the
// CTA has aborted, or after recording a time-out.
template <bool CLUSTER = false>
__device__ bool wait_phase(uint32_t bar, uint32_t parity, Shared *sh, int32_t *err, bool honour_abort = true)
{
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
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

// v[i] <- 2^(v[i]*c2 - r) in place (raw bits) for i in [I0, I0 + 16), z += the
// values as 4 packed pairs of partial sums.
template <int I0>
__device__ __forceinline__ void exp16(uint32_t (&v)[32], uint64_t c2p, uint64_t nrp, uint64_t (&z)[4])
{
#pragma unroll
    for (int i = I0; i < I0 + 16; i += 2) {
        const uint64_t y = fma2(pack2(fv(v[i]), fv(v[i + 1])), c2p, nrp);
        float y0, y1;
        unpack2(y, y0, y1);
        const float e0 = ex2(y0), e1 = ex2(y1);
        v[i] = __float_as_uint(e0);
        v[i + 1] = __float_as_uint(e1);
        z[(i >> 1) & 3] = add2(z[(i >> 1) & 3], pack2(e0, e1));
    }
}

// The softmax side of one CTA for NLD 32-column loads per half row (S = 64*NLD keys).
template <int NLD>
__device__ __forceinline__ void softmax_role(const Geo &g, Shared *sh, int32_t *err, float *__restrict__ scores,
                                             uint32_t tmem, const float2 *xs, float2 *hx, float *red, int ncta,
                                             int T, float c2, int nw, int cid, int nclus, int slice0)
{
    constexpr int S = 64 * NLD;
    constexpr int HALF = 32 * NLD;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sw = warp - 4, q4 = warp & 3, h = sw >> 2;  // TMEM lane quarter, column half
    const int row = 32 * q4 + lane;
    const int sidx = sw * 32 + lane;
    const uint32_t crank = cluster_ctarank();
    const int GW = g.G * g.W;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const uint64_t c2p = pack2(c2, c2);
    const uint32_t xs_u = smem_u32(xs);
    const uint32_t xbytes = (uint32_t)(ncta * kStrip * 8);  // one slot's bytes from all CTAs

    for (int j = 0; j < nw; ++j) {
        const int64_t u = cid + (int64_t)j * nclus;
        uint64_t acc[NLD][16];
#pragma unroll
        for (int k = 0; k < NLD; ++k)
#pragma unroll
            for (int p = 0; p < 16; ++p) acc[k][p] = 0;
        for (int t = 0; t < T; ++t) {
            const int gt = j * T + t, b = gt & 1, slot = gt % kSlots;
            const uint32_t ta = tmem + lane_base + b * 256 + h * HALF;
            // ---- phase A: exponentiate this strip's logits once, keep them in TMEM
            wait_phase(smem_u32(&sh->tfull[b]), (gt >> 1) & 1, sh, err);
            tc_fence_after();
            float rk[NLD];
            float r;
            uint64_t z4[4] = {0, 0, 0, 0};
            // two register sets: chunk k+1 loads, and its maximum is taken, while
            // chunk k is exponentiated (one tcgen05.wait::ld covers all loads in flight)
            uint32_t va[32], vb[32];
            tmem_ld32(ta, va);
            tmem_wait_ld(va);
            r = max32(va) * c2 + kMargin;
            float mn = 0.f;
#pragma unroll
            for (int k = 0; k < NLD; ++k) {
                uint32_t(&cur)[32] = (k & 1) ? vb : va;
                uint32_t(&nxt)[32] = (k & 1) ? va : vb;
                if (k > 0) {
                    if (__any_sync(0xffffffffu, mn > r)) {
                        // rare: a later chunk exceeds the reference; move it up and rescale the sum
                        if (mn > r) {
                            const float rn = mn + kMargin;
                            const float a = ex2(r - rn);
                            const uint64_t ap = pack2(a, a);
#pragma unroll
                            for (int i = 0; i < 4; ++i) z4[i] = fma2(z4[i], ap, 0ull);
                            r = rn;
                        }
                    }
                }
                const uint64_t nrp = pack2(-r, -r);
                if (k + 1 < NLD) tmem_ld32(ta + 32 * (k + 1), nxt);
                exp16<0>(cur, c2p, nrp, z4);
                if (k + 1 < NLD) {
                    tmem_wait_ld_after(nxt, cur);
                    mn = max32(nxt) * c2;
                }
                exp16<16>(cur, c2p, nrp, z4);
                tmem_st32(ta + 32 * k, cur);
                rk[k] = r;
            }
            float z = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float lo, hi;
                unpack2(z4[i], lo, hi);
                z += lo + hi;
            }
            tmem_wait_st();
            // the first chunk of e comes back while the partials are merged and exchanged
            tmem_ld32(ta, va);
            // after a time-out the exchange stops: nothing more is sent and no slot
            // is armed again, so no barrier sees more arrivals than it expects
            const bool live = !*(volatile int *)&sh->abort;
            // the row's two halves merge here; the first half sends the CTA's partial
            float2 *hrow = hx + (gt & 1) * kStrip + row;
            if (h == 1) *hrow = make_float2(r, z);
            named_barrier(2 + q4, 64);
            if (h == 0 && live) {
                const float2 o = *hrow;
                const float rc = fmaxf(r, o.x);
                const float zc = z * ex2(r - rc) + o.y * ex2(o.x - rc);
                const uint32_t xl = xs_u + 8u * (uint32_t)((slot * kMaxCta + (int)crank) * kStrip + row);
                const uint32_t xb = smem_u32(&sh->xfull[slot]);
                for (int c = 0; c < ncta; ++c) st_async_f2(mapa(xl, (uint32_t)c), rc, zc, mapa(xb, (uint32_t)c));
            }
            // ---- phase B: the row's normaliser, then accumulate the weights
            const bool got = live && wait_phase<true>(smem_u32(&sh->xfull[slot]), (uint32_t)(gt / kSlots) & 1u, sh, err);
            float2 pr[kMaxCta];
            float M = -INFINITY;
#pragma unroll
            for (int c = 0; c < kMaxCta; ++c)
                if (c < ncta) {
                    pr[c] = xs[(slot * kMaxCta + c) * kStrip + row];
                    M = fmaxf(M, pr[c].x);
                }
            float Z = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxCta; ++c)
                if (c < ncta) Z = fmaf(pr[c].y, ex2(pr[c].x - M), Z);
            // rows past G*W (the tail of the last strip) add nothing
            const float inv = (got && t * kStrip + row < GW) ? rcp_approx(Z) : 0.f;
            float wk[NLD];
            bool same = true;
#pragma unroll
            for (int k = 0; k < NLD; ++k) same = same && rk[k] == r;
            if (__all_sync(0xffffffffu, same)) {
                const float w = inv * ex2(r - M);
#pragma unroll
                for (int k = 0; k < NLD; ++k) wk[k] = w;
            } else {
#pragma unroll
                for (int k = 0; k < NLD; ++k) wk[k] = inv * ex2(rk[k] - M);
            }
            tmem_wait_ld(va);
#pragma unroll
            for (int k = 0; k < NLD; ++k) {
                uint32_t(&cur)[32] = (k & 1) ? vb : va;
                uint32_t(&nxt)[32] = (k & 1) ? va : vb;
                if (k + 1 < NLD) tmem_ld32(ta + 32 * (k + 1), nxt);
                const uint64_t wp = pack2(wk[k], wk[k]);
#pragma unroll
                for (int p = 0; p < 16; ++p) acc[k][p] = fma2(pack2(fv(cur[2 * p]), fv(cur[2 * p + 1])), wp, acc[k][p]);
                if (k + 1 < NLD) tmem_wait_ld(nxt);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[b]));
            // the slot's next use is strip gt + kSlots; every peer sends it only after
            // this CTA has finished this strip (see the slot count)
            if (sidx == 0 && got) mbar_arrive_expect_tx(smem_u32(&sh->xfull[slot]), xbytes);
        }

        // ---- window done: column sums over the 128 lanes, in a fixed order
        float vals[NLD * 32];
#pragma unroll
        for (int k = 0; k < NLD; ++k)
#pragma unroll
            for (int p = 0; p < 16; ++p) unpack2(acc[k][p], vals[32 * k + 2 * p], vals[32 * k + 2 * p + 1]);
        // butterfly over the warp's lanes: after the round with offset o the lane
        // keeps the half of its range selected by bit o of its lane id
#pragma unroll
        for (int o = 16, n = NLD * 32; o >= 1; o >>= 1, n >>= 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < n / 2; ++i) {
                const float send = upper ? vals[i] : vals[n / 2 + i];
                const float keep = upper ? vals[n / 2 + i] : vals[i];
                vals[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
        // lane l now holds keys NLD*l .. NLD*l + NLD - 1 of its half, summed over its warp's 32 rows.
        // The window's validity, from the same table the producer read (a window
        // with a bad block id or length was not loaded; its scores are zeros).
        int ws_, wl_, wh_;
        window_coords(g, u, ws_, wl_, wh_);
        const int32_t L = g.len[ws_];
        const bool len_ok = L >= g.W && ((int64_t)L + g.bs - 1) / g.bs <= g.bt_stride;
        if (len_ok) {
            const int lb = (L - g.W) / g.bs + sidx;  // at most W/16 + 1 <= 65 blocks per window
            if (lb < (L + g.bs - 1) / g.bs) {
                const int32_t bid = g.bt[(int64_t)ws_ * g.bt_stride + lb];
                if (bid < 0 || bid >= g.num_blocks) sh->wbad[j & 1] = j + 1;
            }
        }
        named_barrier(1, kSoft);
        const int stat = !len_ok ? KARA_EINVAL : *(volatile int *)&sh->wbad[j & 1] == j + 1 ? KARA_EBADBLOCK : 0;
#pragma unroll
        for (int k = 0; k < NLD; ++k) red[q4 * kSlice + h * HALF + NLD * lane + k] = vals[k];
        named_barrier(1, kSoft);
        if (sidx < S) {
            const float sum = ((red[sidx] + red[kSlice + sidx]) + red[2 * kSlice + sidx]) + red[3 * kSlice + sidx];
            const int key = slice0 + sidx;
            if (key < g.C) scores[u * g.C + key] = stat ? 0.f : sum;
        }
        if (stat && sidx == 0) set_err(err, stat);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    score_sp_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap, const Geo g,
                    float *__restrict__ scores, int32_t *err, int ncta, int T, float c2, uint64_t wait_ns, int stall)
{
    using C_ = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *sK = base;                                   // two key buffers
    uint8_t *sQ = sK + 2 * C_::kKBytes;                   // two query stages
    float2 *xs = reinterpret_cast<float2 *>(sQ + 2 * C_::kQBytes);
    float2 *hx = xs + kSlots * kSlotFloats2;              // the halves' partials, by strip parity
    float *red = reinterpret_cast<float *>(hx + 2 * kStrip);
    Shared *sh = reinterpret_cast<Shared *>(red + 4 * kSlice);
    const uint32_t sK_u = smem_u32(sK), sQ_u = smem_u32(sQ);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const int cid = blockIdx.x / ncta, nclus = gridDim.x / ncta;
    const int nw = cid < g.nwin ? (int)((g.nwin - cid + nclus - 1) / nclus) : 0;
    const int slice0 = (int)crank * kSlice;
    const int S = min(kSlice, g.W - slice0);              // keys of this CTA, a multiple of 64

    // -- set-up: barriers, TMEM, exchange slots armed for strips 0 .. kSlots-1
    if (threadIdx.x == 0) {
        sh->abort = 0;
        sh->wait_ns = wait_ns;
        sh->wbad[0] = sh->wbad[1] = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sh->qfull[i]), 1);
            mbar_init(smem_u32(&sh->qempty[i]), 1);
            mbar_init(smem_u32(&sh->kfull[i]), 1);
            mbar_init(smem_u32(&sh->kempty[i]), 1);
            mbar_init(smem_u32(&sh->tfull[i]), 1);
            mbar_init(smem_u32(&sh->tempty[i]), kSoft / 32);
        }
        for (int i = 0; i < kSlots; ++i) mbar_init(smem_u32(&sh->xfull[i]), 1);
        mbar_init(smem_u32(&sh->done), 1);
        fence_mbarrier_init();
        for (int i = 0; i < kSlots; ++i) mbar_arrive_expect_tx(smem_u32(&sh->xfull[i]), (uint32_t)(ncta * kStrip * 8));
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sh->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&qmap);
        prefetch_tmap(&kmap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // every peer's barriers exist before anyone sends to them
    cluster_arrive();
    cluster_wait();
    const uint32_t tmem = sh->tmem_base;

    if (warp >= 4) {
        // ---------------- softmax warpgroups ---------------------------------
        // (the register increase sits in the same branch as the code that uses it)
        reg_alloc<kRegsHigh>();
        const int nld = S / 64;
        if (nld == 4)
            softmax_role<4>(g, sh, err, scores, tmem, xs, hx, red, ncta, T, c2, nw, cid, nclus, slice0);
        else if (nld == 3)
            softmax_role<3>(g, sh, err, scores, tmem, xs, hx, red, ncta, T, c2, nw, cid, nclus, slice0);
        else if (nld == 2)
            softmax_role<2>(g, sh, err, scores, tmem, xs, hx, red, ncta, T, c2, nw, cid, nclus, slice0);
        else
            softmax_role<1>(g, sh, err, scores, tmem, xs, hx, red, ncta, T, c2, nw, cid, nclus, slice0);
    } else {
        reg_dealloc<kRegsLow>();
        if (warp == 0) {
            // ---------------- producer: key slices and query strips by TMA --------
            int issued = 0, kissued = 0;  // query strips, key slices issued
            // Window j's key slice goes into buffer j & 1, one TMA box per (paged
            // block, 64-column atom), a block's 16 rows at 16-row steps; a block
            // id outside the pool reads zeros (the tensor map's bounds) and the
            // softmax warps report the window.
            auto load_k = [&](int j) {
                const int64_t u = cid + (int64_t)j * nclus;
                int s, l, h;
                window_coords(g, u, s, l, h);
                const int32_t L = g.len[s];
                const bool ok = L >= g.W && ((int64_t)L + g.bs - 1) / g.bs <= g.bt_stride;
                const int x0 = L - g.W + slice0;
                const int b0 = ok ? x0 / kBlockRows : 0;
                const int nblk = ok ? (x0 + S - 1) / kBlockRows - b0 + 1 : 0;
                const int32_t myblk = lane < nblk ? g.bt[(int64_t)s * g.bt_stride + b0 + lane] : 0;
                const int kb = j & 1;
                if (lane == 0 && j >= 2) wait_phase(smem_u32(&sh->kempty[kb]), ((j - 2) >> 1) & 1, sh, err);
                __syncwarp();
                const uint32_t bar = smem_u32(&sh->kfull[kb]);
                if (lane == 0 && !stall) mbar_arrive_expect_tx(bar, (uint32_t)(nblk * C_::kAtoms * C_::kBoxBytes));
                for (int i = 0; i < nblk; ++i) {
                    const int32_t blk = __shfl_sync(0xffffffffu, myblk, i);
                    if (lane == 0 && !stall)
#pragma unroll
                        for (int a = 0; a < C_::kAtoms; ++a)
                            tma_load_5d(sK_u + kb * C_::kKBytes + a * kKAtomBytes + i * C_::kBoxBytes, &kmap, bar,
                                        a * 64, 0, h, blk, l);
                }
                kissued = j + 1;
            };
            if (nw > 0) load_k(0);
            for (int j = 0; j < nw; ++j) {
                const int64_t u = cid + (int64_t)j * nclus;
                int s, l, h;
                window_coords(g, u, s, l, h);
                const int row0 = ((s * g.layers + l) * g.hq + h * g.G) * g.W;
                for (int t = 0; t < T; ++t) {
                    const int gt = j * T + t, st = gt & 1;
                    if (lane == 0 && !stall && !*(volatile int *)&sh->abort) {
                        if (wait_phase(smem_u32(&sh->qempty[st]), ((gt >> 1) & 1) ^ 1, sh, err)) {
                            const uint32_t fb = smem_u32(&sh->qfull[st]);
                            mbar_arrive_expect_tx(fb, C_::kQBytes);
#pragma unroll
                            for (int a = 0; a < C_::kAtoms; ++a)
                                tma_load_2d(sQ_u + st * C_::kQBytes + a * C_::kQAtomBytes, &qmap, fb, a * 64,
                                            row0 + t * kStrip);
                            issued = gt + 1;
                            // warm L2 with the strip after next, which all CTAs of the cluster read
                            if (t + 2 < T)
#pragma unroll
                                for (int a = 0; a < C_::kAtoms; ++a)
                                    tma_prefetch_2d(&qmap, a * 64, row0 + (t + 2) * kStrip);
                        }
                    }
                    __syncwarp();
                    // the next window's key slice, once this window's second strip is on its
                    // way: by then the previous window's MMAs, which read that buffer, are done
                    if (t == (T > 1 ? 1 : 0) && j + 1 < nw) load_k(j + 1);
                }
            }
            // drain: every issued copy has landed before this CTA may exit
            if (lane == 0 && !stall) {
                for (int gt = max(0, issued - 2); gt < issued; ++gt)
                    wait_phase(smem_u32(&sh->qfull[gt & 1]), (gt >> 1) & 1, sh, err, false);
                for (int j = max(0, kissued - 2); j < kissued; ++j)
                    wait_phase(smem_u32(&sh->kfull[j & 1]), (j >> 1) & 1, sh, err, false);
            }
            __syncwarp();
        } else if (warp == 1) {
            // ---------------- MMA issuer -----------------------------------------
            const uint32_t idesc = idesc_bf16(128, S);
            if (lane == 0) {
                bool ok = true;
                for (int j = 0; j < nw && ok; ++j) {
                    const int kb = j & 1;
                    // the window's first key sits o rows into the key buffer
                    int s, l, h;
                    window_coords(g, cid + (int64_t)j * nclus, s, l, h);
                    const int32_t L = g.len[s];
                    const int o = L >= g.W ? (L - g.W + slice0) % kBlockRows : 0;
                    ok = wait_phase(smem_u32(&sh->kfull[kb]), (j >> 1) & 1, sh, err);
                    for (int t = 0; t < T && ok; ++t) {
                        const int gt = j * T + t, st = gt & 1;
                        ok = wait_phase(smem_u32(&sh->qfull[st]), (gt >> 1) & 1, sh, err) &&
                             wait_phase(smem_u32(&sh->tempty[st]), ((gt >> 1) & 1) ^ 1, sh, err);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < C_::kKSteps; ++kk) {
                            const int a = kk >> 2, off = (kk & 3) * 32;
                            const uint64_t ad = sdesc_sw128(sQ_u + st * C_::kQBytes + a * C_::kQAtomBytes + off);
                            // the tensor core applies the 128-byte swizzle to absolute shared
                            // addresses, as TMA wrote them, so starting o rows in needs no more
                            const uint64_t bd = sdesc_sw128(sK_u + kb * C_::kKBytes + a * kKAtomBytes + o * 128 + off);
                            mma_bf16(tmem + st * 256, ad, bd, idesc, kk > 0);
                        }
                        mma_commit(smem_u32(&sh->qempty[st]));
                        mma_commit(smem_u32(&sh->tfull[st]));
                    }
                    if (ok) mma_commit(smem_u32(&sh->kempty[kb]));
                }
                // every MMA issued has completed before TMEM is freed
                mma_commit(smem_u32(&sh->done));
                wait_phase(smem_u32(&sh->done), 0, sh, err, false);
            }
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    // no CTA leaves while a peer may still send to its shared memory
    cluster_arrive();
    cluster_wait();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
cudaError_t launch_sp(const Geo &g, float *scores, int32_t *err, cudaStream_t st)
{
    const int ncta = (g.W + kSlice - 1) / kSlice;
    const int T = (g.G * g.W + kStrip - 1) / kStrip;
    const size_t smem = smem_bytes<D>();
    auto fn = tensor_map_encoder();
    if (!fn) return cudaErrorNotSupported;
    // query rows: [n * layers * hq * W][D]
    CUtensorMap qmap;
    {
        const cuuint64_t rows = (cuuint64_t)g.n * g.layers * g.hq * g.W;
        cuuint64_t dims[2] = {(cuuint64_t)D, rows};
        cuuint64_t strides[1] = {(cuuint64_t)D * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)kStrip};
        cuuint32_t estr[2] = {1, 1};
        if (fn(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(g.q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // key pool: (d, slot, kv head, block, layer), strides from the cache description
    CUtensorMap kmap;
    {
        cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)kBlockRows, (cuuint64_t)g.hkv, (cuuint64_t)g.num_blocks,
                              (cuuint64_t)g.layers};
        cuuint64_t strides[4] = {(cuuint64_t)D * 2, (cuuint64_t)g.head_stride * 2, (cuuint64_t)g.block_stride * 2,
                                 (cuuint64_t)g.layer_stride * 2};
        cuuint32_t box[5] = {64, (cuuint32_t)kBlockRows, 1, 1, 1};
        cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        if (fn(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<uint16_t *>(g.k), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    auto kern = score_sp_kernel<D>;
    // the warpgroups' register trade is only safe with the launch count it was sized for
    static int regs[2] = {0, 0};
    int &nreg = regs[D == 128];
    if (nreg == 0) {
        cudaFuncAttributes fa;
        cudaError_t e0 = cudaFuncGetAttributes(&fa, kern);
        if (e0 != cudaSuccess) return e0;
        nreg = fa.numRegs;
    }
    if (nreg != kRegsLaunch) return cudaErrorInvalidKernelImage;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ncta;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // one resident cluster per group of ncta SMs; each walks its share of the windows
    static int resident[2][kMaxCta + 1] = {};
    int &nres = resident[D == 128][ncta];
    if (nres == 0) {
        cfg.gridDim = dim3((unsigned)ncta);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        nres = n;
    }
    const int64_t nclus = g.nwin < nres ? g.nwin : nres;
    cfg.gridDim = dim3((unsigned)(nclus * ncta));
    const float c2 = 1.4426950408889634f / sqrtf((float)D);
    const Stall dbg = debug_stall(kTimeoutNs);
    return cudaLaunchKernelEx(&cfg, kern, qmap, kmap, g, scores, err, ncta, T, c2, dbg.wait_ns, (int)dbg.on);
}

}  // namespace

// The single-pass kernel covers bidirectional scoring with at most kMaxCta key slices.
bool score_sp_supported(const Geo &g) { return !g.causal && g.W <= kSlice * kMaxCta; }

cudaError_t launch_score_sp(const Geo &g, float *scores, int32_t *err, cudaStream_t st)
{
    return g.D == 128 ? launch_sp<128>(g, scores, err, st) : launch_sp<64>(g, scores, err, st);
}

}  // namespace kara
