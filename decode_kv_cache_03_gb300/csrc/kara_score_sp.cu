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
// protected buffer) take part in the normalisation but are not scored.  The
// causal ablation (score_mode KARA_SCORE_CAUSAL) runs the same kernel with
// keys j > i masked out of query i's softmax: their exponentials are 0.
//
// Each logit is computed and exponentiated exactly once:
//
//   * One thread-block cluster per window, one CTA per slice of <= 256 window
//     keys (cluster size ceil(W/256) <= 8).  The key slice comes into shared
//     memory by TMA, one 16-row paged block at a time through a 5-D tensor map
//     over the pool (128-byte swizzled, the tensor core's K-major layout); the
//     window's first key may sit o rows into its block, so the MMA operand
//     starts o rows into the buffer.  The G*W query rows of the window stream
//     through a TMA ring in 128-row strips.
//   * Per strip, S = Q_strip * K_slice^T (M = 128 rows, N = slice) goes into
//     one of two TMEM buffers.
//   * Exponential warps (two per TMEM lane quarter; a thread owns one query row
//     and half of the slice's keys) turn the strip's logits into
//     e = 2^(l2 - r), l2 = <q,k> log2(e)/sqrt(D), written back over S in TMEM,
//     and send their partial sum z = sum e of the row to every CTA of the
//     cluster with st.async (DSMEM, completing bytes on the receiver's
//     mbarrier).  The reference r is common to the cluster: the row position's
//     log-sum-exp two strips earlier in the same window (0 for a window's first
//     two strips), r + log2(sum z), which every CTA derives from the same
//     exchanged partials in the same order (two strips back, that exchange has
//     long completed).  It cancels in e / Z.  So no pass over the logits
//     precedes the exponentials, and the row's normaliser is a plain sum.  A strip whose row total sum_c z_c leaves [2^-88, 2^119] --
//     where the fp32 exponentials could overflow, or lose terms within 2^-30
//     of the row maximum -- marks its window, and an exact CUDA-core kernel
//     recomputes marked windows afterwards (with the usual logit ranges no
//     window is marked).
//   * Accumulating warps (two per lane quarter, half of the keys each) wait
//     for the ncta partials of their row, form Z = sum_c z_c in a fixed order,
//     read e back from TMEM and accumulate e / Z in registers, one fp32
//     accumulator per (row lane, key).  That releases the TMEM buffer for the
//     next strip's MMA.  The exponentials of one strip overlap the exchange
//     and accumulation of the previous one.
//   * After a window's last strip the accumulators are summed across the 32
//     lanes of each warp (a butterfly that leaves each lane whole keys) and
//     across the four lane quarters through shared memory, in a fixed order.
//
// The kernel is persistent: each cluster walks its share of the windows, and
// (up to 4 CTAs per cluster) the next window's key slice loads into the second
// key buffer while the current window is scored; with 5..8 CTAs the exchange
// slots take that room and a slice loads after the previous window's last MMA.
// No W x W matrix and no per-row statistic reaches global memory; every score
// is a deterministic fp32 sum that depends on its own window only.  Warp roles (640
// threads): warps 0..7 exponentials (two per lane quarter, one per half of the
// keys), 8..15 accumulation, 16 query-strip TMA, 17 TMEM allocation and MMAs
// (one lane), 18 key-slice TMA (it also reads the window's length and block ids
// once and publishes the first key's row offset and the window's validity in
// shared memory), 19 idle; the warpgroups trade registers so the accumulating
// warps hold 128 accumulators each.  Every wait is bounded;
// on time-out the CTA records KARA_ETIMEOUT and stops waiting, still draining
// what it has in flight.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "kara_common.cuh"
#include "kara_sm100.cuh"

namespace kara {

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

using namespace ptx;

constexpr int kSlice = 256;    // keys per CTA
constexpr int kStrip = 128;    // query rows per strip
constexpr int kMaxCta = 8;     // CTAs per cluster: W <= 2048
constexpr int kSlots = 4;      // exchange slots (strips in flight between CTAs)
constexpr int kExpW = 8;       // exponential warps: two per TMEM lane quarter (column halves)
constexpr int kAcc = 256;      // accumulating threads: two per TMEM lane
constexpr int kAccW0 = kExpW;  // first accumulating warp
constexpr int kCtlW0 = kExpW + kAcc / 32;    // control warps: query TMA, MMA, key TMA, idle
constexpr int kThreads = 32 * (kCtlW0 + 4);  // five warpgroups
// Registers per thread: at launch (65536 / 640 rounded down to the allocation
// granule of 8, what ptxas assigns under the launch bounds), then after the
// warpgroups trade registers.  The trade must add up:
// 256 * kRegsExp + 256 * kRegsAcc + 128 * kRegsCtl == 640 * kRegsLaunch.
constexpr int kRegsLaunch = 96;
constexpr uint32_t kRegsExp = 40;
constexpr uint32_t kRegsAcc = 176;
constexpr uint32_t kRegsCtl = 48;
static_assert(256 * kRegsExp + 256 * kRegsAcc + 128 * kRegsCtl == kThreads * kRegsLaunch,
              "register trade must add up");
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr uint64_t kDrainNs = 20000ull;  // landing time allowed to DSMEM stores after a time-out
constexpr int kBlockRows = 16;                         // rows of a paged block
constexpr int kSliceBlocks = kSlice / kBlockRows + 1;  // blocks a slice can touch (17)
constexpr int kKAtomBytes = kSliceBlocks * kBlockRows * 128;  // one 64-column atom of a key buffer
// Window statuses in flight: window j + kWinRing is loaded only after the
// accumulating warps have finished window j, even with one strip per window.
constexpr int kWinRing = 8;
// A row's sum of exponentials relative to its reference must lie here for the
// fp32 exponentials to be exact to rounding: above, the largest could
// overflow; below, terms within 2^-30 of the row maximum could flush to zero.
constexpr float kSumLo = 3.2311742677852644e-27f;   // 2^-88
constexpr float kSumHi = 6.6461399789245794e+35f;   // 2^119

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
    uint64_t tfull[2];               // S of a strip is in TMEM
    uint64_t eready[2];              // its exponentials are back in TMEM
    uint64_t tempty[2];              // the TMEM buffer may be written again
    uint64_t xfull[kSlots];          // exchange slots
    uint64_t wfull[kWinRing];        // a window's status is published
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    uint64_t wait_ns;
    int unsafe[2];                   // 1 + index of the last window (by parity) whose sums left the safe range
    int koff[2];                     // row of the window's first key in each key buffer
    int wstat[kWinRing];             // a window's status: 0, KARA_EINVAL or KARA_EBADBLOCK
};

// An instantiation of the kernel covers clusters of up to MAXC CTAs: 4 (W <=
// 1024) or 8 (W <= 2048).  Its exchange slot holds the partial sums of MAXC
// CTAs for each row, one per column half.  Up to 4 CTAs there are two key-slice
// buffers (the next window's slice loads while the current one is scored);
// with 8 the larger slots leave room for one, and a window's slice loads after
// the previous window's last MMA.
template <int MAXC>
constexpr int kSlotF = MAXC * 2 * kStrip;
template <int MAXC>
constexpr int kKeyBufs = MAXC > 4 ? 1 : 2;

template <int D, int MAXC>
size_t smem_bytes()
{
    using C_ = Cfg<D>;
    const size_t need = 1024 + (size_t)kKeyBufs<MAXC> * C_::kKBytes + 2 * (size_t)C_::kQBytes
                      + (size_t)kSlots * kSlotF<MAXC> * 4 + 4 * kSlice * 4 + sizeof(Shared);
    // more than half of the SM's shared memory: a second CTA never shares the
    // SM and waits in tcgen05.alloc for the TMEM this persistent one holds
    const size_t floor_ = 120 * 1024;
    return need > floor_ ? need : floor_;
}

// Bounded wait on an mbarrier phase.  Returns false (without waiting) once the
// CTA has aborted, or after recording a time-out.
// POLL: test without suspending (for the MMA issuer, whose reaction is on the
// critical path).
template <bool CLUSTER = false, bool POLL = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, Shared *sh, int32_t *err,
                                           bool honour_abort = true)
{
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (CLUSTER ? mbar_try_wait_cluster(bar, parity)
                    : POLL ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity))
            return true;
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

// Row total of an exchange slot: the partial sums added in (CTA, half) order,
// so every CTA of the cluster (and both warp roles) gets the same value.
template <int MAXC>
__device__ __forceinline__ float slot_total(const float *xs, int slot, int ncta, int row)
{
    float Z = xs[slot * kSlotF<MAXC> + row] + xs[slot * kSlotF<MAXC> + kStrip + row];
#pragma unroll
    for (int c = 1; c < MAXC; ++c)
        if (c < ncta)
            Z += xs[slot * kSlotF<MAXC> + (2 * c) * kStrip + row] + xs[slot * kSlotF<MAXC> + (2 * c + 1) * kStrip + row];
    return Z;
}

__device__ __forceinline__ bool in_safe_range(float Z) { return Z >= kSumLo && Z <= kSumHi; }  // NaN: false

// v[i] <- 2^(v[i]*c2 - r) in place (raw bits) for the 8 values, z += them as
// 2 packed pairs of partial sums.
__device__ __forceinline__ void exp8(uint32_t (&v)[8], uint64_t c2p, uint64_t nrp, uint64_t (&z)[2])
{
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const uint64_t y = fma2(pack2(fv(v[i]), fv(v[i + 1])), c2p, nrp);
        float y0, y1;
        unpack2(y, y0, y1);
        const float e0 = ex2(y0), e1 = ex2(y1);
        v[i] = __float_as_uint(e0);
        v[i + 1] = __float_as_uint(e1);
        z[(i >> 1) & 1] = add2(z[(i >> 1) & 1], pack2(e0, e1));
    }
}

// exp8 for a chunk that straddles the causal diagonal: value e (key j0 + e) is
// kept where e <= lim (the key is at or before the row's query) and is 0 past it.
__device__ __forceinline__ void exp8_masked(uint32_t (&v)[8], uint64_t c2p, uint64_t nrp, uint64_t (&z)[2], int lim)
{
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const uint64_t y = fma2(pack2(fv(v[i]), fv(v[i + 1])), c2p, nrp);
        float y0, y1;
        unpack2(y, y0, y1);
        const float e0 = i <= lim ? ex2(y0) : 0.f, e1 = i + 1 <= lim ? ex2(y1) : 0.f;
        v[i] = __float_as_uint(e0);
        v[i + 1] = __float_as_uint(e1);
        z[(i >> 1) & 1] = add2(z[(i >> 1) & 1], pack2(e0, e1));
    }
}

// Exponential warps: two per TMEM lane quarter, a thread per query row of the
// strip and half (32 * NLD) of the slice's keys.
template <int NLD, int MAXC, bool CAUSAL>
__device__ __forceinline__ void exp_role(const Geo &g, Shared *sh, int32_t *err, uint32_t tmem, const float *xs,
                                         int ncta, int T, float c2, int nw, int slice0)
{
    constexpr int NCH = 4 * NLD;  // 8-column chunks of this warp's half
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q4 = warp & 3, eh = warp >> 2;
    const int row = 32 * q4 + lane;
    const uint32_t crank = cluster_ctarank();
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const uint64_t c2p = pack2(c2, c2);
    const uint32_t xs_u = smem_u32(xs);
    for (int j = 0; j < nw; ++j) {
        // references of this row position for even and odd strips, the same in
        // every CTA of the cluster; 0 for a window's first two strips, so a
        // window's scores do not depend on the windows scored before it
        float rr[2] = {0.f, 0.f};
        for (int t = 0; t < T; ++t) {
            const int gt = j * T + t, b = gt & 1, slot = gt & (kSlots - 1);
            // the row total of strip gt - 2 of the same window moves that strip's
            // reference to the row's log2-sum-exp (an out-of-range total, which
            // marks the window, or a missing one after a time-out leaves it where
            // it was; once the CTA has aborted, the slots' phases no longer follow
            // the strips)
            if (t > 1) {
                const int ps = (gt - 2) & (kSlots - 1);
                if (wait_phase(smem_u32(&sh->xfull[ps]), (uint32_t)((gt - 2) / kSlots) & 1u, sh, err) &&
                    !*(volatile int *)&sh->abort) {
                    const float Z = slot_total<MAXC>(xs, ps, ncta, row);
                    if (in_safe_range(Z)) rr[b] += __log2f(Z);
                }
            }
            const float r = rr[b];
            const uint32_t ta = tmem + lane_base + b * 256 + eh * (32 * NLD);
            wait_phase(smem_u32(&sh->tfull[b]), (gt >> 1) & 1, sh, err);
            __syncwarp();  // the TMEM accesses below are warp-collective
            tc_fence_after();
            uint64_t z2[2] = {0, 0};
            const uint64_t nrp = pack2(-r, -r);
            // the row's query position minus this warp's first key in the window
            // (causal masking only)
            const int qdiff = CAUSAL ? (t * kStrip + row) % g.W - (slice0 + eh * (32 * NLD)) : 0;
            {
                // two 8-column register sets: chunk c+1 loads while chunk c is
                // exponentiated (one tcgen05.wait::ld covers all loads in flight);
                // the two warps of a lane quarter interleave on the SMSP
                uint32_t ua[8], ub[8];
                tmem_ld8(ta, ua);
                tmem_wait_ld8(ua);
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    uint32_t(&cur)[8] = (c & 1) ? ub : ua;
                    uint32_t(&nxt)[8] = (c & 1) ? ua : ub;
                    if (c + 1 < NCH) tmem_ld8(ta + 8 * (c + 1), nxt);
                    if (CAUSAL) {
                        // keys after the row's query weigh 0 (a select per element,
                        // cheaper than branching on the chunk)
                        exp8_masked(cur, c2p, nrp, z2, qdiff - 8 * c);
                    } else {
                        exp8(cur, c2p, nrp, z2);
                    }
                    tmem_st8(ta + 8 * c, cur);
                    if (c + 1 < NCH) tmem_wait_ld8(nxt);
                }
            }
            float z = 0.f;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                float lo, hi;
                unpack2(z2[i], lo, hi);
                z += lo + hi;
            }
            // the row's partial goes out first (it does not depend on the TMEM
            // stores); after a time-out the exchange stops: nothing more is sent
            if (!*(volatile int *)&sh->abort) {
                const uint32_t xl = xs_u + 4u * (uint32_t)(slot * kSlotF<MAXC> + (2 * (int)crank + eh) * kStrip + row);
                const uint32_t xb = smem_u32(&sh->xfull[slot]);
                for (int c = 0; c < ncta; ++c) st_async_f32(mapa(xl, (uint32_t)c), z, mapa(xb, (uint32_t)c));
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh->eready[b]));
        }
    }
}

// Accumulating warps: two per TMEM lane quarter, a thread per query row of the
// strip and half (NLD 32-column loads) of the slice's keys.
template <int NLD, int MAXC, bool CAUSAL>
__device__ __forceinline__ void acc_role(const Geo &g, Shared *sh, int32_t *err, float *__restrict__ scores,
                                         uint8_t *__restrict__ marks, uint32_t tmem, const float *xs, float *red,
                                         int ncta, int T, int nw, int cid, int nclus, int slice0)
{
    constexpr int S = 64 * NLD;
    constexpr int HALF = 32 * NLD;
    constexpr int NC = 2 * NLD;  // 16-column chunks of this thread's half
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int aw = warp - kAccW0, q4 = warp & 3, h = aw >> 2;  // TMEM lane quarter, column half
    const int row = 32 * q4 + lane;
    const int aidx = aw * 32 + lane;
    const int GW = g.G * g.W;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const uint32_t xbytes = (uint32_t)(ncta * 2 * kStrip * 4);

    for (int j = 0; j < nw; ++j) {
        const int64_t u = cid + (int64_t)j * nclus;
        uint64_t acc[NC][8];
        bool bad = false;  // a row total of this window left the safe range
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int p = 0; p < 8; ++p) acc[k][p] = 0;
        for (int t = 0; t < T; ++t) {
            const int gt = j * T + t, b = gt & 1, slot = gt & (kSlots - 1);
            const uint32_t ta = tmem + lane_base + b * 256 + h * HALF;
            wait_phase(smem_u32(&sh->eready[b]), (gt >> 1) & 1, sh, err);
            __syncwarp();  // the TMEM accesses below are warp-collective
            tc_fence_after();
            // the first two chunks of e come back while the partials are awaited
            uint32_t va[16], vb[16];
            tmem_ld16(ta, va);
            tmem_ld16(ta + 16, vb);
            // (the complete-tx of the partials' st.async makes them visible to the
            // threads that see the phase complete).  Once the CTA has aborted, a
            // slot's phase parity no longer tells which strip it belongs to: the
            // partials are not used and the slot is not armed again (an extra
            // arrival on a barrier whose phase is still pending would over-arrive).
            const bool got = wait_phase(smem_u32(&sh->xfull[slot]), (uint32_t)(gt / kSlots) & 1u, sh, err) &&
                             !*(volatile int *)&sh->abort;
            const float Z = slot_total<MAXC>(xs, slot, ncta, row);
            // rows past G*W (the tail of the last strip) add nothing; a row total
            // out of the safe range marks the window for the exact recompute
            const bool live = got && t * kStrip + row < GW;
            bad |= live && !in_safe_range(Z);
            // (the reciprocal on the FMA pipe: the special-function unit is busy
            // with the exponential warps' stream)
            const float w = (live && in_safe_range(Z)) ? rcp_newton(Z) : 0.f;
            const uint64_t wp = pack2(w, w);
            tmem_wait_ld16x2(va, vb);
#pragma unroll
            for (int k = 0; k < NC; k += 2) {
                // chunks k, k+1 are in va, vb; k+2, k+3 load into them once consumed
#pragma unroll
                for (int p = 0; p < 8; ++p) acc[k][p] = fma2(pack2(fv(va[2 * p]), fv(va[2 * p + 1])), wp, acc[k][p]);
                if (k + 2 < NC) tmem_ld16(ta + 16 * (k + 2), va);
#pragma unroll
                for (int p = 0; p < 8; ++p)
                    acc[k + 1][p] = fma2(pack2(fv(vb[2 * p]), fv(vb[2 * p + 1])), wp, acc[k + 1][p]);
                if (k + 3 < NC) tmem_ld16(ta + 16 * (k + 3), vb);
                if (k + 3 < NC) tmem_wait_ld16x2(va, vb);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[b]));
            // the slot's next use is strip gt + kSlots; every peer sends it only after
            // this CTA has released the buffer of strip gt + kSlots - 2
            if (aidx == 0 && got) mbar_arrive_expect_tx(smem_u32(&sh->xfull[slot]), xbytes);
        }

        // ---- window done: column sums over the 128 lanes, in a fixed order.
        // One 32-key chunk at a time: a butterfly over the warp's lanes (after the
        // round with offset o a lane keeps the half of its range selected by bit o
        // of its lane id) leaves lane l with key 32k + l summed over the warp's 32
        // rows; the four lane quarters are added through shared memory below.
        if (bad) *(volatile int *)&sh->unsafe[j & 1] = j + 1;
        named_barrier(1, kAcc);  // the previous window's sums have been read
#pragma unroll
        for (int k = 0; k < NLD; ++k) {
            float vals[32];
#pragma unroll
            for (int p = 0; p < 16; ++p) unpack2(acc[2 * k + (p >> 3)][p & 7], vals[2 * p], vals[2 * p + 1]);
#pragma unroll
            for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < n / 2; ++i) {
                    const float send = upper ? vals[i] : vals[n / 2 + i];
                    const float keep = upper ? vals[n / 2 + i] : vals[i];
                    vals[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            red[q4 * kSlice + h * HALF + 32 * k + lane] = vals[0];
        }
        // The window's validity, as the key producer found it in the same table it
        // loaded from (a window with a bad block id or length was not loaded; its
        // scores are zeros).
        const bool wok = wait_phase(smem_u32(&sh->wfull[j & (kWinRing - 1)]), (uint32_t)(j / kWinRing) & 1u, sh, err);
        named_barrier(1, kAcc);
        const int stat = wok ? *(volatile int *)&sh->wstat[j & (kWinRing - 1)] : 0;
        if (aidx < S) {
            const float sum = ((red[aidx] + red[kSlice + aidx]) + red[2 * kSlice + aidx]) + red[3 * kSlice + aidx];
            const int key = slice0 + aidx;
            if (key < g.C) scores[u * g.C + key] = stat ? 0.f : sum;
        }
        if (stat && aidx == 0) set_err(err, stat);
        // a row total of this window left the safe range (every CTA of the cluster
        // sees the same totals); the exact kernel recomputes marked windows
        if (aidx == 0 && !stat && *(volatile int *)&sh->unsafe[j & 1] == j + 1) marks[u] = 1;
    }
}

template <int D, int MAXC, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    score_sp_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap, const Geo g,
                    float *__restrict__ scores, uint8_t *__restrict__ marks, int32_t *err, int ncta, int T, float c2,
                    uint64_t wait_ns, int stall)
{
    using C_ = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *sK = base;                                   // two key buffers
    constexpr int nkb = kKeyBufs<MAXC>;
    uint8_t *sQ = sK + nkb * C_::kKBytes;                 // two query stages
    float *xs = reinterpret_cast<float *>(sQ + 2 * C_::kQBytes);
    float *red = xs + kSlots * kSlotF<MAXC>;
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
        sh->unsafe[0] = sh->unsafe[1] = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sh->qfull[i]), 1);
            mbar_init(smem_u32(&sh->qempty[i]), 1);
            mbar_init(smem_u32(&sh->kfull[i]), 1);
            mbar_init(smem_u32(&sh->kempty[i]), 1);
            mbar_init(smem_u32(&sh->tfull[i]), 1);
            mbar_init(smem_u32(&sh->eready[i]), kExpW);
            mbar_init(smem_u32(&sh->tempty[i]), kAcc / 32);
        }
        for (int i = 0; i < kSlots; ++i) mbar_init(smem_u32(&sh->xfull[i]), 1);
        for (int i = 0; i < kWinRing; ++i) mbar_init(smem_u32(&sh->wfull[i]), 1);
        mbar_init(smem_u32(&sh->done), 1);
        fence_mbarrier_init();
        for (int i = 0; i < kSlots; ++i) mbar_arrive_expect_tx(smem_u32(&sh->xfull[i]), (uint32_t)(ncta * 2 * kStrip * 4));
    }
    if (warp == kCtlW0 + 1) {
        tmem_alloc(smem_u32(&sh->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kCtlW0 && lane == 0) {
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
    const int nld = S / 64;

    // (each warpgroup's register change sits in the same branch as the code that uses it)
    if (warp < kAccW0) {
        // ---------------- exponentials --------------------------------------
        reg_dealloc<kRegsExp>();
        if (nld == 4)
            exp_role<4, MAXC, CAUSAL>(g, sh, err, tmem, xs, ncta, T, c2, nw, slice0);
        else if (nld == 3)
            exp_role<3, MAXC, CAUSAL>(g, sh, err, tmem, xs, ncta, T, c2, nw, slice0);
        else if (nld == 2)
            exp_role<2, MAXC, CAUSAL>(g, sh, err, tmem, xs, ncta, T, c2, nw, slice0);
        else
            exp_role<1, MAXC, CAUSAL>(g, sh, err, tmem, xs, ncta, T, c2, nw, slice0);
    } else if (warp < kCtlW0) {
        // ---------------- accumulation ---------------------------------------
        reg_alloc<kRegsAcc>();
        if (nld == 4)
            acc_role<4, MAXC, CAUSAL>(g, sh, err, scores, marks, tmem, xs, red, ncta, T, nw, cid, nclus, slice0);
        else if (nld == 3)
            acc_role<3, MAXC, CAUSAL>(g, sh, err, scores, marks, tmem, xs, red, ncta, T, nw, cid, nclus, slice0);
        else if (nld == 2)
            acc_role<2, MAXC, CAUSAL>(g, sh, err, scores, marks, tmem, xs, red, ncta, T, nw, cid, nclus, slice0);
        else
            acc_role<1, MAXC, CAUSAL>(g, sh, err, scores, marks, tmem, xs, red, ncta, T, nw, cid, nclus, slice0);
    } else {
        reg_dealloc<kRegsCtl>();
        if (warp == kCtlW0) {
            // ---------------- query strips by TMA ----------------------------------
            int issued = 0;
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
                }
            }
            // drain: every issued copy has landed before this CTA may exit
            if (lane == 0 && !stall)
                for (int gt = max(0, issued - 2); gt < issued; ++gt)
                    wait_phase(smem_u32(&sh->qfull[gt & 1]), (gt >> 1) & 1, sh, err, false);
            __syncwarp();
        } else if (warp == kCtlW0 + 2) {
            // ---------------- key slices by TMA ------------------------------------
            // Window j's key slice goes into buffer j & 1, one TMA box per (paged
            // block, 64-column atom), a block's 16 rows at 16-row steps; a block
            // id outside the pool reads zeros (the tensor map's bounds).  The
            // window's length and all its block ids are read here once: the first
            // key's row offset goes to the MMA issuer with the buffer, the window's
            // status to the accumulating warps.
            int kissued = 0;
            for (int j = 0; j < nw; ++j) {
                const int64_t u = cid + (int64_t)j * nclus;
                int s, l, h;
                window_coords(g, u, s, l, h);
                const int32_t L = g.len[s];
                const bool ok = L >= g.W && ((int64_t)L + g.bs - 1) / g.bs <= g.bt_stride;
                const int32_t *btr = g.bt + (int64_t)s * g.bt_stride;
                // every block of the window (at most W/16 + 1 <= 65), as each CTA of
                // the cluster must reach the same verdict
                bool bad = false;
                if (ok)
                    for (int lb = (L - g.W) / g.bs + lane; lb < (L + g.bs - 1) / g.bs; lb += 32) {
                        const int32_t bid = btr[lb];
                        bad |= bid < 0 || bid >= g.num_blocks;
                    }
                bad = __any_sync(0xffffffffu, bad);
                const int x0 = L - g.W + slice0;
                const int b0 = ok ? x0 / kBlockRows : 0;
                const int nblk = ok ? (x0 + S - 1) / kBlockRows - b0 + 1 : 0;
                const int32_t myblk = lane < nblk ? btr[b0 + lane] : 0;
                // buffer kb's use j / nkb waits for the MMAs of its previous use
                const int kb = j % nkb;
                int go = 0;
                if (lane == 0) {
                    if (j >= nkb) wait_phase(smem_u32(&sh->kempty[kb]), (uint32_t)(j / nkb - 1) & 1u, sh, err);
                    sh->koff[kb] = ok ? x0 % kBlockRows : 0;
                    sh->wstat[j & (kWinRing - 1)] = !ok ? KARA_EINVAL : bad ? KARA_EBADBLOCK : 0;
                    mbar_arrive(smem_u32(&sh->wfull[j & (kWinRing - 1)]));
                    // after a time-out nothing more is loaded: the buffer may still be
                    // read, and its barrier still waits for the previous load
                    go = !stall && !*(volatile int *)&sh->abort;
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (go) {
                    const uint32_t bar = smem_u32(&sh->kfull[kb]);
                    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nblk * C_::kAtoms * C_::kBoxBytes));
                    for (int i = 0; i < nblk; ++i) {
                        const int32_t blk = __shfl_sync(0xffffffffu, myblk, i);
                        if (lane == 0)
#pragma unroll
                            for (int a = 0; a < C_::kAtoms; ++a)
                                tma_load_5d(sK_u + kb * C_::kKBytes + a * kKAtomBytes + i * C_::kBoxBytes, &kmap,
                                            bar, a * 64, 0, h, blk, l);
                    }
                    kissued = j + 1;
                }
            }
            if (lane == 0 && !stall)
                for (int j = max(0, kissued - nkb); j < kissued; ++j)
                    wait_phase(smem_u32(&sh->kfull[j % nkb]), (uint32_t)(j / nkb) & 1u, sh, err, false);
            __syncwarp();
        } else if (warp == kCtlW0 + 1) {
            // ---------------- MMA issuer -----------------------------------------
            const uint32_t idesc = idesc_bf16(128, S);
            if (lane == 0) {
                bool ok = true;
                for (int j = 0; j < nw && ok; ++j) {
                    const int kb = j % nkb;
                    ok = wait_phase(smem_u32(&sh->kfull[kb]), (uint32_t)(j / nkb) & 1u, sh, err);
                    // the window's first key sits o rows into the key buffer
                    const int o = *(volatile int *)&sh->koff[kb];
                    for (int t = 0; t < T && ok; ++t) {
                        const int gt = j * T + t, st = gt & 1;
                        ok = wait_phase(smem_u32(&sh->qfull[st]), (gt >> 1) & 1, sh, err) &&
                             wait_phase<false, true>(smem_u32(&sh->tempty[st]), ((gt >> 1) & 1) ^ 1, sh, err);
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
    // After a time-out nothing waited for a peer's last partials, which may
    // still be in flight to this CTA's shared memory: give them time to land.
    if (*(volatile int *)&sh->abort) {
        if (threadIdx.x == 0) {
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < kDrainNs) {
            }
        }
        __syncthreads();
    }
    if (warp == kCtlW0 + 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Exact scores of the marked windows on the CUDA cores (fp32; the row maximum
// found before any exponential): each CTA walks the marks of its share of the
// windows and computes the few marked ones.  Unmarked windows cost one byte read.
constexpr int kFbThreads = 256;
constexpr int kFbMaxGW = 8192;

__global__ void __launch_bounds__(kFbThreads) exact_kernel(const Geo g, float *__restrict__ scores,
                                                           const uint8_t *__restrict__ marks)
{
    __shared__ float lse[kFbMaxGW];
    const float sc = 1.f / sqrtf((float)g.D);
    for (int64_t u = blockIdx.x; u < g.nwin; u += gridDim.x) {
        if (!marks[u]) continue;
        int s, l, h;
        window_coords(g, u, s, l, h);
        const int32_t L = g.len[s];
        const int ws = L - g.W, GW = g.G * g.W;
        const int32_t *btr = g.bt + (int64_t)s * g.bt_stride;
        const uint16_t *qw = g.q + (((int64_t)s * g.layers + l) * g.hq + (int64_t)h * g.G) * g.W * g.D;
        auto key = [&](int j) { const int x = ws + j; return g.k + pool_off(g, l, btr[x / g.bs], h, x % g.bs); };
        auto bf = [](uint16_t x) { return __uint_as_float((uint32_t)x << 16); };
        auto dot = [&](const uint16_t *a, const uint16_t *b) {
            float acc = 0.f;
            for (int d = 0; d < g.D; ++d) acc = fmaf(bf(a[d]), bf(b[d]), acc);
            return acc * sc;
        };
        // pass 1: per query row, log-sum-exp over all W keys (maximum first); with
        // the causal mask, over the keys at or before the row's query position
        for (int r = threadIdx.x; r < GW; r += blockDim.x) {
            const uint16_t *q = qw + (int64_t)r * g.D;
            const int nk = g.causal ? r % g.W + 1 : g.W;
            float m = -INFINITY;
            for (int j = 0; j < nk; ++j) m = fmaxf(m, dot(q, key(j)));
            float z = 0.f;
            for (int j = 0; j < nk; ++j) z += expf(dot(q, key(j)) - m);
            lse[r] = m + logf(z);
        }
        __syncthreads();
        // pass 2: per compressible key, the sum of the rows' probabilities
        for (int j = threadIdx.x; j < g.C; j += blockDim.x) {
            const uint16_t *k = key(j);
            float acc = 0.f;
            for (int r = 0; r < GW; ++r)
                if (!g.causal || r % g.W >= j) acc += expf(dot(qw + (int64_t)r * g.D, k) - lse[r]);
            scores[u * g.C + j] = acc;
        }
        __syncthreads();
    }
}

// Clusters of ncta CTAs of the scorer that fit on the device at once (one CTA
// per SM), from the occupancy query, cached per shape.  Sets the kernel's
// dynamic shared memory limit, which the query and the launch both need.
template <int D, int MAXC, bool CAUSAL>
cudaError_t resident_clusters(int ncta, int *out)
{
    auto kern = score_sp_kernel<D, MAXC, CAUSAL>;
    const size_t smem = smem_bytes<D, MAXC>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    static int resident[kMaxCta + 1] = {};
    int &nres = resident[ncta];
    if (nres == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.gridDim = dim3((unsigned)ncta);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = ncta;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        nres = n;
    }
    *out = nres;
    return cudaSuccess;
}

template <int D, int MAXC, bool CAUSAL>
cudaError_t launch_sp(const Geo &g, float *scores, uint8_t *marks, int32_t *err, cudaStream_t st)
{
    const int ncta = (g.W + kSlice - 1) / kSlice;
    const int T = (g.G * g.W + kStrip - 1) / kStrip;
    const size_t smem = smem_bytes<D, MAXC>();
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

    auto kern = score_sp_kernel<D, MAXC, CAUSAL>;
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
    int nres = 0;
    cudaError_t e = resident_clusters<D, MAXC, CAUSAL>(ncta, &nres);
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
    const int64_t nclus = g.nwin < nres ? g.nwin : nres;
    cfg.gridDim = dim3((unsigned)(nclus * ncta));
    const float c2 = 1.4426950408889634f / sqrtf((float)D);
    const Stall dbg = debug_stall(kTimeoutNs);
    e = cudaMemsetAsync(marks, 0, (size_t)g.nwin, st);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, kern, qmap, kmap, g, scores, marks, err, ncta, T, c2, dbg.wait_ns, (int)dbg.on);
    if (e != cudaSuccess) return e;
    const unsigned fb_blocks = (unsigned)(g.nwin < 1184 ? g.nwin : 1184);
    exact_kernel<<<fb_blocks, kFbThreads, 0, st>>>(g, scores, marks);
    return cudaGetLastError();
}

}  // namespace

// The single-pass kernel covers bidirectional scoring with at most kMaxCta key slices.
bool score_sp_supported(const Geo &g) { return g.W <= kSlice * kMaxCta && g.G * g.W <= kFbMaxGW; }

// resident_clusters of the instantiation that covers clusters of ncta CTAs.
static cudaError_t resident_for(int D, int ncta, int *nres)
{
    if (ncta <= 4)
        return D == 128 ? resident_clusters<128, 4, false>(ncta, nres) : resident_clusters<64, 4, false>(ncta, nres);
    return D == 128 ? resident_clusters<128, 8, false>(ncta, nres) : resident_clusters<64, 8, false>(ncta, nres);
}

// SMs the single-pass scorer leaves without a CTA of its own while it runs on
// batch g (0 when it does not cover g or a query fails): other work can use
// them meanwhile.
int score_idle_sms(const Geo &g)
{
    if (!score_sp_supported(g) || g.nwin == 0) return 0;
    const int ncta = (g.W + kSlice - 1) / kSlice;
    int nres = 0, dev = 0, sms = 0;
    if (resident_for(g.D, ncta, &nres) != cudaSuccess) return 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    const int64_t used = (g.nwin < nres ? g.nwin : nres) * (int64_t)ncta;
    return sms > used ? (int)(sms - used) : 0;
}

// Resident clusters of the single-pass scorer for batch g (0 when it does not cover g).
int score_resident_clusters(const Geo &g)
{
    if (!score_sp_supported(g)) return 0;
    const int ncta = (g.W + kSlice - 1) / kSlice;
    int nres = 0;
    if (resident_for(g.D, ncta, &nres) != cudaSuccess) return 0;
    return nres;
}

// Scratch of the single-pass path: one mark byte per window.
size_t score_sp_scratch_bytes(const Geo &g) { return g.W <= kSlice * kMaxCta ? align256((size_t)g.nwin) : 0; }

// Scratch of the scoring path: one mark byte per window.
size_t score_scratch_bytes(const Geo &g) { return score_sp_scratch_bytes(g); }

cudaError_t launch_score_sp(const Geo &g, float *scores, void *scratch, int32_t *err, cudaStream_t st);

// Every shape the entry points accept (W <= 2048, G * W <= 8192, bidirectional
// or causal) is scored in one pass over the logits.
cudaError_t launch_score(const Geo &g, float *scores, void *scratch, int32_t *err, cudaStream_t st)
{
    if (g.nwin == 0) return cudaSuccess;
    if (!score_sp_supported(g)) return cudaErrorInvalidValue;
    return launch_score_sp(g, scores, scratch, err, st);
}

cudaError_t launch_score_sp(const Geo &g, float *scores, void *scratch, int32_t *err, cudaStream_t st)
{
    uint8_t *marks = static_cast<uint8_t *>(scratch);
    const int ncta = (g.W + kSlice - 1) / kSlice;
    if (g.causal) {
        if (ncta <= 4)
            return g.D == 128 ? launch_sp<128, 4, true>(g, scores, marks, err, st)
                              : launch_sp<64, 4, true>(g, scores, marks, err, st);
        return g.D == 128 ? launch_sp<128, 8, true>(g, scores, marks, err, st)
                          : launch_sp<64, 8, true>(g, scores, marks, err, st);
    }
    if (ncta <= 4)
        return g.D == 128 ? launch_sp<128, 4, false>(g, scores, marks, err, st)
                          : launch_sp<64, 4, false>(g, scores, marks, err, st);
    return g.D == 128 ? launch_sp<128, 8, false>(g, scores, marks, err, st)
                      : launch_sp<64, 8, false>(g, scores, marks, err, st);
}

}  // namespace kara
