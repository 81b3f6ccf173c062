// kara_compact_static: the compaction entry point for callers that cannot
// obtain device memory when compaction runs.
//
// A serving engine typically hands all free HBM to its KV-cache pool at
// start-up, and some embed this library where no device allocator is
// reachable at all; such callers can pass their inputs and outputs but no
// workspace.  This variant keeps the one piece of scratch that compaction
// needs -- the per-sequence page plan -- in a fixed array compiled into the
// library instead.  It runs the same plan, copy and commit kernels as
// kara_compact; only where the plan lives differs.
#include "kara_common.cuh"

using namespace kara;

// The plan of every sequence of a call (32 bytes each).  Every GPU that loads
// the library holds this array until the process exits.  All calls share it.
static __device__ __align__(256) SeqPlan g_static_plan[KARA_STATIC_MAX_SEQS];

namespace {

// Device address of g_static_plan in the current context.  In host code the
// array's name denotes a host-side stand-in, not device memory, so the kernels
// are given this looked-up address.  It is looked up on every call (a host-side
// query that allocates nothing): a cached address would outlive the context
// it came from, e.g. across cudaDeviceReset.
kara_status static_plan(SeqPlan **out)
{
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_static_plan) != cudaSuccess || !addr) return KARA_ECUDA;
    *out = static_cast<SeqPlan *>(addr);
    return KARA_OK;
}

}  // namespace

extern "C" kara_status kara_compact_static(const kara_cache *c, const kara_params *p, const kara_batch *b,
                                           const int32_t *kept, const int32_t *fresh, int64_t n_fresh,
                                           int32_t *freed, int32_t *new_len, int32_t *err,
                                           kara_stream_t stream)
{
    const Range range("kara_compact_static");
    Geo g;
    kara_status st = geo_from_args(c, p, b, &g);
    if (st != KARA_OK) return st;
    if (g.n > KARA_STATIC_MAX_SEQS) return KARA_EUNSUPPORTED;
    if (g.n == 0) return KARA_OK;
    if (!kept || !new_len || !err || n_fresh < 0 || (n_fresh > 0 && !fresh) || !freed) return KARA_EINVAL;
    SeqPlan *plan = nullptr;
    st = static_plan(&plan);
    if (st != KARA_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    // plan_kernel writes every entry [0, n) that compact_kernel and commit_kernel
    // read, so what an earlier call left in the array is never seen.
    cudaError_t e = launch_plan(g, n_fresh, plan, err, s);
    if (e == cudaSuccess) e = launch_compact(g, plan, kept, fresh, n_fresh, err, s);
    if (e == cudaSuccess) e = launch_commit(g, plan, fresh, freed, new_len, b->block_table, err, s);
    return e == cudaSuccess ? KARA_OK : KARA_ECUDA;
}
