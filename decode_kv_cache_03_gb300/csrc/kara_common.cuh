// Shared device/host helpers of the Kara sm_103a library (internal header).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "kara.h"

namespace kara {

// Failure-detection knob for tests.  With KARA_DEBUG_STALL=1 in the
// environment, the kernels that stage data through shared memory issue no
// copies at all, so every wait on data runs out -- after wait_ns = 1 ms
// instead of the normal limit -- and the call reports KARA_ETIMEOUT.  Nothing
// is in flight when those waits give up, and the waits that drain in-flight
// work keep the normal limit.
struct Stall {
    int32_t on;
    uint64_t wait_ns;
};

// Named range on the host timeline of a profiler (NVTX; a no-op when no tool
// is attached), one per public call that launches work.
struct Range {
    explicit Range(const char *name);
    ~Range();
    Range(const Range &) = delete;
    Range &operator=(const Range &) = delete;
};

inline Stall debug_stall(uint64_t normal_ns)
{
    const char *v = getenv("KARA_DEBUG_STALL");
    const bool on = v && v[0] == '1' && v[1] == 0;
    return Stall{on ? 1 : 0, on ? 1000000ull : normal_ns};
}

// Per-sequence plan produced on the device by plan_kernel (summary section 3:
// the trailing blocks of a sequence are rebuilt and the old ones released).
struct SeqPlan {
    int32_t L;        // cached length
    int32_t ws;       // window start = L - W
    int32_t p0;       // first rebuilt logical block = ws / bs
    int32_t Lnew;     // L - C + R
    int32_t n_new;    // fresh blocks taken
    int32_t n_old;    // old tail blocks released
    int32_t off_new;  // offset of this sequence's ids in the fresh list
    int32_t off_old;  // offset in the freed list
};

// Geometry shared by every kernel of one call.
struct Geo {
    const uint16_t *k;    // bf16 pools as raw bits
    const uint16_t *v;
    int64_t layer_stride, block_stride, head_stride;
    int32_t layers, num_blocks, hkv, hq, G, D, bs;
    int32_t W, B, C, K, R;
    float lambda;
    int32_t n, bt_stride;
    const int32_t *len;
    const int32_t *bt;
    const uint16_t *q;
    int64_t nwin;         // n * layers * hkv
    int32_t causal;       // score_mode == KARA_SCORE_CAUSAL
};

__device__ __forceinline__ void set_err(int32_t *err, int code)
{
    if (err) atomicCAS(err, 0, code);
}

// Window u -> (sequence, layer, kv head).
__device__ __forceinline__ void window_coords(const Geo &g, int64_t u, int &s, int &l, int &h)
{
    h = (int)(u % g.hkv);
    l = (int)((u / g.hkv) % g.layers);
    s = (int)(u / ((int64_t)g.hkv * g.layers));
}

// Offset (elements) of a pool row; blk must already be range-checked.
__device__ __forceinline__ int64_t pool_off(const Geo &g, int l, int32_t blk, int h, int slot)
{
    return (int64_t)l * g.layer_stride + (int64_t)blk * g.block_stride + (int64_t)h * g.head_stride
         + (int64_t)slot * g.D;
}

__host__ __device__ __forceinline__ size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Host-side argument checks of the entry points; fills the geometry of a call.
kara_status geo_from_args(const kara_cache *c, const kara_params *p, const kara_batch *b, Geo *g);

// Launchers (each returns the launch error, if any).
cudaError_t launch_plan(const Geo &g, int64_t n_fresh, SeqPlan *plan, int32_t *err, cudaStream_t st);
cudaError_t launch_compact(const Geo &g, const SeqPlan *plan, const int32_t *kept, const int32_t *fresh,
                           int64_t n_fresh, int32_t *err, cudaStream_t st);
// The two halves of launch_compact: the fresh-id check of a whole batch, and the
// kept-row check plus the copy of a batch or of a group of its sequences (plan
// then points at the group's first entry; offsets into fresh stay the batch's).
cudaError_t launch_fresh_check(const Geo &g, const SeqPlan *plan, const int32_t *fresh, int64_t n_fresh,
                               int32_t *err, cudaStream_t st);
cudaError_t launch_kept_copy(const Geo &g, const SeqPlan *plan, const int32_t *kept, const int32_t *fresh,
                             int64_t n_fresh, int32_t *err, cudaStream_t st);
cudaError_t launch_commit(const Geo &g, const SeqPlan *plan, const int32_t *fresh, int32_t *freed,
                          int32_t *new_len, int32_t *bt, const int32_t *err, cudaStream_t st);
cudaError_t launch_select(int64_t nwin, int C, int K, int R, float lambda, int mode, int chunk, const float *scores,
                          int32_t *cand, int32_t *kept, cudaStream_t st);
size_t score_scratch_bytes(const Geo &g);
cudaError_t launch_decode(const kara_cache *c, int32_t layer, int32_t n, const int32_t *len, const int32_t *bt,
                          int32_t bt_stride, const void *q, float *out, void *ws, int32_t *err, cudaStream_t st);
size_t decode_workspace_bytes(const kara_cache *c, int32_t n, int32_t bt_stride);
cudaError_t launch_qring_compact(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                 const int32_t *kept, int32_t *err, cudaStream_t st);
cudaError_t launch_qring_append(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                const void *q_new, cudaStream_t st);
int decode_max_splits(int32_t bt_stride, int32_t block_size);
cudaError_t launch_score(const Geo &g, float *scores, void *scratch, int32_t *err, cudaStream_t st);
// SMs the single-pass scorer leaves idle on batch g, and its resident clusters
// (both 0 when the single-pass kernel does not cover g).
int score_idle_sms(const Geo &g);
int score_resident_clusters(const Geo &g);

}  // namespace kara
