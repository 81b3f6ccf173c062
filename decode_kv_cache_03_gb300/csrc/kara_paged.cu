// Page plan, gather-compaction and block-table commit for paged K/V pools.
//
// Follows the gist.science summary of Kara (arXiv 2607.01237), section
// "3. KvLLM Framework and Periodic Compression": Kara runs on PagedAttention
// blocks, compresses the trailing blocks of the selected sequences and frees
// memory.  The retained rows of each window are packed, in order, into fresh
// blocks supplied by the caller; the old tail blocks are released only after
// every copy is done and only if no error was recorded.
#include "kara_common.cuh"

namespace kara {
namespace {

constexpr int kPlanThreads = 1024;

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

// Exclusive scan of one int per thread over the block; *total gets the sum.
__device__ int block_excl_scan(int v, int *scratch /* >= 33 ints */, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = warp_incl_scan(v);
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = lane < nw ? scratch[lane] : 0;
        int xi = warp_incl_scan(x);
        if (lane < nw) scratch[lane] = xi - x;
        if (lane == 31) scratch[32] = xi;
    }
    __syncthreads();
    int r = scratch[warp] + incl - v;
    *total = scratch[32];
    __syncthreads();
    return r;
}

// One block computes every sequence's plan and the offsets of its fresh and
// freed ids (exclusive prefix sums in sequence order).
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(Geo g, int64_t n_fresh, SeqPlan *plan,
                                                            int32_t *err)
{
    __shared__ int scratch[33];
    __shared__ long long carry_new, carry_old;
    if (threadIdx.x == 0) { carry_new = 0; carry_old = 0; }
    __syncthreads();
    for (int base = 0; base < g.n; base += blockDim.x) {
        const int s = base + threadIdx.x;
        SeqPlan p;
        p.L = 0; p.ws = 0; p.p0 = -1; p.Lnew = 0; p.n_new = 0; p.n_old = 0;
        if (s < g.n) {
            const int32_t L = g.len[s];
            p.L = L;
            p.Lnew = L;
            const bool ok = L >= g.W && ((int64_t)L + g.bs - 1) / g.bs <= g.bt_stride;
            if (!ok) {
                set_err(err, KARA_EINVAL);
            } else {
                p.ws = L - g.W;
                p.p0 = p.ws / g.bs;
                p.Lnew = p.ws + g.R + g.B;
                p.n_old = (L + g.bs - 1) / g.bs - p.p0;
                p.n_new = (p.Lnew + g.bs - 1) / g.bs - p.p0;
            }
        }
        int tot_new, tot_old;
        const int ex_new = block_excl_scan(p.n_new, scratch, &tot_new);
        const int ex_old = block_excl_scan(p.n_old, scratch, &tot_old);
        p.off_new = (int32_t)(carry_new + ex_new);
        p.off_old = (int32_t)(carry_old + ex_old);
        if (s < g.n) plan[s] = p;
        __syncthreads();
        if (threadIdx.x == 0) { carry_new += tot_new; carry_old += tot_old; }
        __syncthreads();
    }
    if (threadIdx.x == 0 && carry_new > n_fresh) set_err(err, KARA_ENOBLOCKS);
}

// The inputs the copy must not run with, checked before it writes anything:
// the rewrite fills fresh blocks while the batch's old blocks are still read,
// so a consumed fresh id must be new.
//   - fresh_check_kernel: every fresh id the plan consumes, fresh[i] for
//     i < total_new, against the earlier consumed ids and against every entry
//     below ceil(L/bs) of every table of the batch (a block the batch keeps or
//     still reads), as raw values: a match records KARA_EDUPBLOCK.  An id
//     outside [0, num_blocks) records KARA_EBADBLOCK, which a match overrides.
//   - kept_check_kernel: each window's kept row must be strictly increasing in
//     [0, C) (Top-K and Token2Chunk produce ascending positions): KARA_EINVAL.
// Each probe value (a consumed fresh id or a table entry) is compared with the
// consumed fresh ids through tiles staged in shared memory: no scratch memory,
// and the work is (total_new + n * bt_stride) * total_new comparisons.
constexpr int kChkThreads = 256;
constexpr int kChkProbes = 4;     // probe values per thread
constexpr int kChkTile = 2048;    // fresh ids per shared-memory tile

__device__ __forceinline__ void record_dup(int32_t *err)
{
    if (atomicCAS(err, 0, KARA_EDUPBLOCK) == KARA_EBADBLOCK) atomicCAS(err, KARA_EBADBLOCK, KARA_EDUPBLOCK);
}

__global__ void __launch_bounds__(kChkThreads) fresh_check_kernel(Geo g, const SeqPlan *__restrict__ plan,
                                                                  const int32_t *__restrict__ fresh,
                                                                  int64_t n_fresh, int32_t *err)
{
    __shared__ int32_t tile[kChkTile];
    const SeqPlan last = plan[g.n - 1];
    const int64_t F = (int64_t)last.off_new + last.n_new;  // fresh ids the plan consumes
    if (F > n_fresh) return;                                // KARA_ENOBLOCKS is recorded
    const int64_t P = F + (int64_t)g.n * g.bt_stride;       // probes: consumed ids, then table slots
    int32_t v[kChkProbes];
    int64_t lim[kChkProbes];                                // compare with fresh[j], j < lim
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kChkProbes; ++k) {
        const int64_t p = ((int64_t)blockIdx.x * kChkProbes + k) * kChkThreads + threadIdx.x;
        v[k] = 0;
        lim[k] = 0;
        if (p < F) {
            v[k] = fresh[p];
            lim[k] = p;
            bad |= v[k] < 0 || v[k] >= g.num_blocks;
        } else if (p < P) {
            const int64_t q = p - F;
            const int s = (int)(q / g.bt_stride), lb = (int)(q % g.bt_stride);
            const int64_t L = g.len[s];
            if (L > 0 && lb < (L + g.bs - 1) / g.bs) {
                v[k] = g.bt[q];
                lim[k] = F;
            }
        }
    }
    bool dup = false;
    for (int64_t t0 = 0; t0 < F; t0 += kChkTile) {
        const int n = (int)min((int64_t)kChkTile, F - t0);
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += kChkThreads) tile[i] = fresh[t0 + i];
        __syncthreads();
        for (int i = 0; i < n; ++i) {
            const int32_t f = tile[i];
#pragma unroll
            for (int k = 0; k < kChkProbes; ++k) dup |= f == v[k] && t0 + i < lim[k];
        }
    }
    if (bad) atomicCAS(err, 0, KARA_EBADBLOCK);
    if (dup) record_dup(err);
}

__global__ void __launch_bounds__(kChkThreads) kept_check_kernel(int64_t n, int R, int C,
                                                                 const int32_t *__restrict__ kept, int32_t *err)
{
    for (int64_t i = (int64_t)blockIdx.x * kChkThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kChkThreads) {
        const int r = (int)(i % R);
        const int32_t k = kept[i];
        if (k < 0 || k >= C || (r > 0 && kept[i - 1] >= k)) set_err(err, KARA_EINVAL);
    }
}

// One block per (window, K|V): copies o + R + B rows of D bf16 with 16-byte
// vector loads/stores, old rows read through the old table, new rows written
// into the sequence's fresh blocks.
template <int D>
__global__ void __launch_bounds__(256) compact_kernel(Geo g, const SeqPlan *__restrict__ plan,
                                                      const int32_t *__restrict__ kept,
                                                      const int32_t *__restrict__ fresh,
                                                      int64_t n_fresh, int32_t *err)
{
    constexpr int CPR = D * 2 / 16;  // 16-byte chunks per row
    constexpr int UNROLL = 4;
    // nothing is written once an earlier kernel (plan, checks) recorded an error
    if (*(volatile const int32_t *)err != 0) return;
    const int64_t u = blockIdx.x >> 1;
    const int which = blockIdx.x & 1;
    int s, l, h;
    window_coords(g, u, s, l, h);
    const SeqPlan p = plan[s];
    if (p.p0 < 0 || (int64_t)p.off_new + p.n_new > n_fresh) return;  // error already recorded
    const uint16_t *pool_src = which ? g.v : g.k;
    uint16_t *pool_dst = const_cast<uint16_t *>(pool_src);
    const int rows = p.Lnew - p.p0 * g.bs;
    const int32_t *kp = kept + u * g.R;
    const int32_t *bt_row = g.bt + (int64_t)s * g.bt_stride;
    const int32_t *fr = fresh + p.off_new;
    const int total = rows * CPR;
    for (int base = threadIdx.x; base < total; base += blockDim.x * UNROLL) {
        uint4 val[UNROLL];
        int64_t dst[UNROLL];
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
            dst[k] = -1;
            const int idx = base + k * blockDim.x;
            if (idx >= total) continue;
            const int r = idx / CPR, c = idx % CPR;
            const int xn = p.p0 * g.bs + r;
            int xo;
            if (xn < p.ws) {
                xo = xn;
            } else if (xn < p.ws + g.R) {
                const int kk = kp[xn - p.ws];
                if (kk < 0 || kk >= g.C) { set_err(err, KARA_EINVAL); continue; }
                xo = p.ws + kk;
            } else {
                xo = p.L - g.B + (xn - p.ws - g.R);
            }
            const int32_t ob = bt_row[xo / g.bs];
            const int32_t nb = fr[xn / g.bs - p.p0];
            if (ob < 0 || ob >= g.num_blocks || nb < 0 || nb >= g.num_blocks) {
                set_err(err, KARA_EBADBLOCK);
                continue;
            }
            val[k] = *reinterpret_cast<const uint4 *>(pool_src + pool_off(g, l, ob, h, xo % g.bs) + c * 8);
            dst[k] = pool_off(g, l, nb, h, xn % g.bs) + c * 8;
        }
#pragma unroll
        for (int k = 0; k < UNROLL; ++k)
            if (dst[k] >= 0) *reinterpret_cast<uint4 *>(pool_dst + dst[k]) = val[k];
    }
}

// One warp per sequence: release the old tail, install the fresh ids, set the
// new length -- only when no error was recorded by any earlier kernel.
__global__ void __launch_bounds__(256) commit_kernel(Geo g, const SeqPlan *__restrict__ plan,
                                                     const int32_t *__restrict__ fresh,
                                                     int32_t *freed, int32_t *new_len, int32_t *bt,
                                                     const int32_t *err)
{
    const int s = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= g.n) return;
    const int32_t e = *err;
    const SeqPlan p = plan[s];
    if (e != 0 || p.p0 < 0) {
        if (lane == 0) new_len[s] = g.len[s];
        return;
    }
    int32_t *row = bt + (int64_t)s * g.bt_stride + p.p0;
    for (int t = lane; t < p.n_old; t += 32) {
        const int32_t old = row[t];
        freed[p.off_old + t] = old;
        row[t] = t < p.n_new ? fresh[p.off_new + t] : -1;
    }
    if (lane == 0) new_len[s] = p.Lnew;
}

}  // namespace

cudaError_t launch_plan(const Geo &g, int64_t n_fresh, SeqPlan *plan, int32_t *err, cudaStream_t st)
{
    plan_kernel<<<1, kPlanThreads, 0, st>>>(g, n_fresh, plan, err);
    return cudaGetLastError();
}

// The fresh-id check of the whole batch (before any copy of any group).
cudaError_t launch_fresh_check(const Geo &g, const SeqPlan *plan, const int32_t *fresh, int64_t n_fresh,
                               int32_t *err, cudaStream_t st)
{
    if (g.nwin == 0) return cudaSuccess;
    const int64_t probes = n_fresh + (int64_t)g.n * g.bt_stride;
    const int64_t per = (int64_t)kChkThreads * kChkProbes;
    const int64_t nb = (probes + per - 1) / per;
    if (nb > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    fresh_check_kernel<<<(unsigned)nb, kChkThreads, 0, st>>>(g, plan, fresh, n_fresh, err);
    return cudaGetLastError();
}

// The kept-row check, then the copy (which runs only if no error was recorded).
cudaError_t launch_kept_copy(const Geo &g, const SeqPlan *plan, const int32_t *kept, const int32_t *fresh,
                             int64_t n_fresh, int32_t *err, cudaStream_t st)
{
    const int64_t blocks = g.nwin * 2;
    if (blocks == 0) return cudaSuccess;
    const int64_t nk = g.nwin * g.R;
    const int64_t kb = (nk + kChkThreads - 1) / kChkThreads;
    kept_check_kernel<<<(unsigned)(kb < 4096 ? kb : 4096), kChkThreads, 0, st>>>(nk, g.R, g.C, kept, err);
    if (g.D == 128)
        compact_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(g, plan, kept, fresh, n_fresh, err);
    else
        compact_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(g, plan, kept, fresh, n_fresh, err);
    return cudaGetLastError();
}

// The checks, then the copy (which runs only if no error was recorded).
cudaError_t launch_compact(const Geo &g, const SeqPlan *plan, const int32_t *kept, const int32_t *fresh,
                           int64_t n_fresh, int32_t *err, cudaStream_t st)
{
    const cudaError_t e = launch_fresh_check(g, plan, fresh, n_fresh, err, st);
    return e == cudaSuccess ? launch_kept_copy(g, plan, kept, fresh, n_fresh, err, st) : e;
}

cudaError_t launch_commit(const Geo &g, const SeqPlan *plan, const int32_t *fresh, int32_t *freed,
                          int32_t *new_len, int32_t *bt, const int32_t *err, cudaStream_t st)
{
    if (g.n == 0) return cudaSuccess;
    const int blocks = (g.n + 7) / 8;
    commit_kernel<<<blocks, 256, 0, st>>>(g, plan, fresh, freed, new_len, bt, err);
    return cudaGetLastError();
}

}  // namespace kara
