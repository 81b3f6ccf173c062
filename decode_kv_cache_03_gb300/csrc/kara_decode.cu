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
// The work is HBM-bound (about 2.5 FLOP per byte of K and V).  Flash-decoding
// layout: one CTA per (sequence, KV head, split of kSplit keys).  A producer
// warp streams the split's K blocks, then its V blocks, into a ring of
// shared-memory stages by TMA: one (block, KV head) slice of 16 rows per
// stage, as 64-dim halves in the 128-byte swizzled layout, so many blocks are
// in flight per SM without holding registers.  Four consumer warps take one
// block each.  The G query heads of a KV head share every key, so both
// contractions of a block are small bf16 matrix products on the warp-level
// tensor-core MMA (m16n8k16, fp32 accumulators), the operands read from the
// swizzled stage with ldmatrix, free of bank conflicts:
//   logits   S^T[16 keys][8 heads]  = K_blk[16][D] . Q^T[D][8]
//   outputs  O^T[D][8 heads]       += V_blk^T[D][16] . P^T[16][8]
// The weights P are fp32; each enters the second product as the sum of two
// bf16 terms (hi = rn(p), lo = rn(p - hi)), so its relative error is about
// 2^-17, as good as the fp32 sums around it.  The tensor cores here only
// save issue slots: on the CUDA cores the same work took about 46 warp
// instructions per key and the consumers, not HBM, set the pace; here it
// takes about 4.  Between the two products, the softmax of the split runs in
// shared memory.  A second kernel combines the splits of each (sequence, head)
// in a fixed order, so the result is deterministic.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kara_common.cuh"
#include "kara_sm100.cuh"

namespace kara {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();  // defined beside the scoring kernel

namespace {

constexpr int kSplit = 1024;        // keys per CTA
constexpr int kBlk = 16;            // tokens per cache block (the supported block size)
constexpr int kBlocks = kSplit / kBlk;
constexpr int kNC = 4;              // consumer warps
constexpr int kDecThreads = 32 * (1 + kNC);
constexpr int kStages = 8;          // ring of (block, head) slices in flight
constexpr int kHalf = kBlk * 64 * 2;  // bytes of one 64-dim half of a slice: 16 swizzled 128-byte rows
constexpr int kLs = kSplit + 8;     // row stride of the logits (floats): the weight fragments load conflict-free
constexpr uint64_t kDecTimeoutNs = 1000000000ull;  // 1 s: a stage normally lands in microseconds
// Blocks go to the consumer warps round-robin and stage waits are by phase
// parity, which tells only two neighbouring phases apart: a warp may wait for
// use j of a stage only after it has seen use j - kStages complete, so both
// uses must be its own.
static_assert(kStages % kNC == 0, "each stage is reused by the same consumer warp");

struct DecodeArgs {
    int32_t layer, num_blocks, hkv, hq, G, bs;
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

// ---- warp-level tensor-core operands -------------------------------------------
// Four 8x8 bf16 tiles from shared memory; lanes 8i..8i+7 give the row
// addresses of tile i, which lands in r[i].
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// The same, each tile transposed on the way.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// d += A[16x16] . B[16x8], bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (lo, hi) rounded to nearest-even bf16, lo in the low half.
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// p = hi + lo + O(2^-17 p), both bf16 pairs; p - hi is exact in fp32.
__device__ __forceinline__ void split_bf16x2(float2 p, uint32_t &hi, uint32_t &lo)
{
    hi = bf16x2(p.x, p.y);
    lo = bf16x2(p.x - __uint_as_float(hi << 16), p.y - __uint_as_float(hi & 0xffff0000u));
}

// Dynamic shared memory: 1 KB of alignment slack, ring[kStages] of slices
// (each [D/64 halves][16 rows][128 B], 128-byte swizzled), logit[G][kLs] fp32
// (logits, then weights, then the consumers' partial outputs), DecShared.
// Four CTAs per SM (32 slices in flight) up to G = 5 at D = 128; wider
// groups' logits leave room for three.
template <int D, int G>
constexpr int dec_min_blocks() { return D == 128 && G >= 6 ? 3 : 4; }

template <int D, int G>
constexpr size_t dec_smem_bytes()
{
    return 1024 + (size_t)kStages * kBlk * D * 2 + sizeof(float) * G * kLs + sizeof(DecShared);
}

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, dec_min_blocks<D, G>())
    decode_split_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const DecodeArgs a, int32_t *err)
{
    constexpr int BB = kBlk * D * 2;  // bytes of one (block, head) slice
    constexpr int NH = D / 64;        // 64-dim halves of a row
    constexpr int KS = D / 16;        // k-steps of the logits = 16-dim tiles of the outputs
    static_assert(G <= 8, "heads per group: one n8 tile");
    static_assert(kNC * D <= kLs, "partial outputs fit in the logit area");
    extern __shared__ uint8_t dsm_raw[];
    // the swizzle pattern repeats every 1024 bytes and is taken from the address
    uint8_t *ring = dsm_raw + ((1024u - (ptx::smem_u32(dsm_raw) & 1023u)) & 1023u);
    float *logit = reinterpret_cast<float *>(ring + kStages * BB);  // [G][kLs]
    DecShared *sh = reinterpret_cast<DecShared *>(logit + G * kLs);

    // launched as a programmatic dependent of whatever precedes it on the
    // stream (the previous call's merge, or the compaction that rewrote the
    // table): nothing global is read before that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
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
            ptx::prefetch_tmap(&kmap);
            ptx::prefetch_tmap(&vmap);
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
                    const CUtensorMap *m = j < nb ? &kmap : &vmap;
#pragma unroll
                    for (int h = 0; h < NH; ++h)
                        ptx::tma_load_5d(ptx::smem_u32(ring + st * BB + h * kHalf), m, fb, h * 64, 0, g, blk, a.layer);
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
    // MMA fragment coordinates: row group r8 = lane / 4, thread tq = lane % 4.
    const int cw = warp - 1, ctid = threadIdx.x - 32;
    const int r8 = lane >> 2, tq = lane & 3;

    // Logits' B operand Q^T[16 dims][8 heads]: head r8, dims 16ks + 2tq + {0, 1}
    // and + 8; heads past G are zero.
    uint32_t qb[KS][2];
    {
        const uint32_t *qh =
            reinterpret_cast<const uint32_t *>(a.q + ((int64_t)s * a.hq + g * G + min(r8, G - 1)) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qb[ks][0] = r8 < G ? __ldg(qh + ks * 8 + tq) : 0u;
            qb[ks][1] = r8 < G ? __ldg(qh + ks * 8 + 4 + tq) : 0u;
        }
    }

    // ---- logits.  A = K rows of the block: tile i of ldmatrix = (rows 8(i&1).., dims +8(i>>1));
    // in the swizzled stage, 16-byte chunk c of row t sits at chunk c ^ (t & 7)
    const int kt = lane & 15, kc = lane >> 4;
    for (int i = cw; i < nb; i += kNC) {
        const int st = i % kStages;
        if (!dwait(ptx::smem_u32(&sh->full[st]), (i / kStages) & 1, sh, err, a.wait_ns)) break;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        if (sh->bad[st] == 0) {
            const uint32_t sb = ptx::smem_u32(ring + st * BB) + kt * 128;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t af[4];
                ldsm_x4(sb + (ks >> 2) * kHalf + ((((ks & 3) * 2 + kc) ^ (kt & 7)) << 4), af);
                mma_16816(c, af, qb[ks][0], qb[ks][1]);
            }
        }
        // the MMAs have consumed the block's bytes: hand the stage back
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sh->empty[st]));
        // c = S^T at (key r8, heads 2tq, 2tq+1) and (key r8 + 8, same heads); a zero row gives logit 0
        const int x = i * kBlk + r8, h0 = 2 * tq;
        if (h0 < G) {
            if (x < nk) logit[h0 * kLs + x] = c[0] * a.scale2;
            if (x + 8 < nk) logit[h0 * kLs + x + 8] = c[2] * a.scale2;
        }
        if (h0 + 1 < G) {
            if (x < nk) logit[(h0 + 1) * kLs + x] = c[1] * a.scale2;
            if (x + 8 < nk) logit[(h0 + 1) * kLs + x + 8] = c[3] * a.scale2;
        }
    }
    ptx::named_barrier(1, kNC * 32);

    // ---- softmax of each head over the split (warp cw: heads cw, cw + kNC) -------
    for (int h = cw; h < G; h += kNC) {
        float *lr = logit + h * kLs;
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

    // ---- weighted sum.  A = V^T (dims x keys) by transposing ldmatrix: tile i =
    // (keys 8(i>>1).., dims +8(i&1)); B = P^T (keys x heads) from the weights
    float acc[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
    const int vt = (lane & 7) + ((lane >> 4) << 3), vc = (lane >> 3) & 1;
    for (int i = cw; i < nb; i += kNC) {
        const int j = nb + i, st = j % kStages;
        if (!dwait(ptx::smem_u32(&sh->full[st]), (j / kStages) & 1, sh, err, a.wait_ns)) break;
        if (sh->bad[st] == 0) {
            // weights of head r8 for keys 2tq, 2tq+1 and 2tq+8, 2tq+9 of the block, as bf16 hi + lo
            uint32_t bh0 = 0u, bl0 = 0u, bh1 = 0u, bl1 = 0u;
            if (r8 < G) {
                const float *w = logit + r8 * kLs + i * kBlk + 2 * tq;
                split_bf16x2(*reinterpret_cast<const float2 *>(w), bh0, bl0);
                split_bf16x2(*reinterpret_cast<const float2 *>(w + 8), bh1, bl1);
            }
            // rows of the last block past the end hold whatever the block held
            // (NaN included): their halves of the fragments are zeroed
            const int tmax = min(kBlk, nk - i * kBlk);
            uint32_t m_lo = 0xffffffffu, m_hi = 0xffffffffu;
            if (tmax < kBlk) {
                m_lo = (2 * tq < tmax ? 0x0000ffffu : 0u) | (2 * tq + 1 < tmax ? 0xffff0000u : 0u);
                m_hi = (2 * tq + 8 < tmax ? 0x0000ffffu : 0u) | (2 * tq + 9 < tmax ? 0xffff0000u : 0u);
            }
            const uint32_t sb = ptx::smem_u32(ring + st * BB) + vt * 128;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                uint32_t af[4];
                ldsm_x4_t(sb + (mt >> 2) * kHalf + ((((mt & 3) * 2 + vc) ^ (vt & 7)) << 4), af);
                af[0] &= m_lo, af[1] &= m_lo, af[2] &= m_hi, af[3] &= m_hi;
                mma_16816(acc[mt], af, bh0, bh1);
                mma_16816(acc[mt], af, bl0, bl1);
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sh->empty[st]));
    }
    // every consumer is done with the weights: the logit area takes the partial
    // outputs red[kNC][G][D], summed below over the warps in a fixed order
    ptx::named_barrier(1, kNC * 32);
    float *red = logit;
    {
        const int h0 = 2 * tq;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const int d = mt * 16 + r8;  // acc[mt] = O^T at (dims d, d + 8; heads h0, h0 + 1)
            if (h0 < G) {
                red[(cw * G + h0) * D + d] = acc[mt][0];
                red[(cw * G + h0) * D + d + 8] = acc[mt][2];
            }
            if (h0 + 1 < G) {
                red[(cw * G + h0 + 1) * D + d] = acc[mt][1];
                red[(cw * G + h0 + 1) * D + d + 8] = acc[mt][3];
            }
        }
    }
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
    // the merge kernel may be scheduled once every CTA of this grid got here
    // or exited; it still waits for this grid's completion before reading
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// out[s][h] = sum_sp part * 2^(m_sp - M) / sum_sp z_sp * 2^(m_sp - M), splits in order.
// Launched as a programmatic dependent of the split kernel: its launch overlaps
// the split grid's last CTAs, and it waits here until that grid has completed
// and its writes are visible.  It lets the next call's split kernel launch as
// it finishes.
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeArgs a)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
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
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Tensor map over one pool, (d, slot, kv head, block, layer) with the cache's
// strides; a box is one 64-dim half of a (block, head) slice, 128-byte swizzled.
cudaError_t pool_map(CUtensorMap *m, const void *pool, const kara_cache *c)
{
    auto fn = tensor_map_encoder();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[5] = {(cuuint64_t)c->head_dim, (cuuint64_t)kBlk, (cuuint64_t)c->num_kv_heads,
                          (cuuint64_t)c->num_blocks, (cuuint64_t)c->num_layers};
    cuuint64_t strides[4] = {(cuuint64_t)c->head_dim * 2, (cuuint64_t)c->head_stride * 2,
                             (cuuint64_t)c->block_stride * 2, (cuuint64_t)c->layer_stride * 2};
    cuuint32_t box[5] = {64, (cuuint32_t)kBlk, 1, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(pool), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

// A tensor map depends only on the pool's address, shape and strides: the
// library keeps the last pair it encoded (static storage, under a lock), so a
// decode loop over the layers of one cache encodes them once.
struct PoolMaps {
    CUtensorMap km, vm;
    const void *k, *v;
    int64_t layer_stride, block_stride, head_stride;
    int32_t num_layers, num_blocks, num_kv_heads, head_dim;
    bool valid;
};

bool same_pools(const PoolMaps &m, const kara_cache *c)
{
    return m.valid && m.k == c->k && m.v == c->v && m.layer_stride == c->layer_stride &&
           m.block_stride == c->block_stride && m.head_stride == c->head_stride && m.num_layers == c->num_layers &&
           m.num_blocks == c->num_blocks && m.num_kv_heads == c->num_kv_heads && m.head_dim == c->head_dim;
}

cudaError_t pool_maps(const kara_cache *c, CUtensorMap *km, CUtensorMap *vm)
{
    static std::mutex mu;
    static PoolMaps m{};
    std::lock_guard<std::mutex> lock(mu);
    if (!same_pools(m, c)) {
        m.valid = false;
        cudaError_t e = pool_map(&m.km, c->k, c);
        if (e == cudaSuccess) e = pool_map(&m.vm, c->v, c);
        if (e != cudaSuccess) return e;
        m.k = c->k, m.v = c->v;
        m.layer_stride = c->layer_stride, m.block_stride = c->block_stride, m.head_stride = c->head_stride;
        m.num_layers = c->num_layers, m.num_blocks = c->num_blocks, m.num_kv_heads = c->num_kv_heads;
        m.head_dim = c->head_dim;
        m.valid = true;
    }
    *km = m.km;
    *vm = m.vm;
    return cudaSuccess;
}

template <int D, int G>
cudaError_t launch_split_g(const CUtensorMap &km, const CUtensorMap &vm, const DecodeArgs &a, dim3 grid,
                           int32_t *err, cudaStream_t st)
{
    const size_t smem = dec_smem_bytes<D, G>();
    auto kern = decode_split_kernel<D, G>;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, km, vm, a, err);
}

template <int D>
cudaError_t launch_split(const CUtensorMap &km, const CUtensorMap &vm, const DecodeArgs &a, dim3 grid, int32_t *err,
                         cudaStream_t st)
{
    switch (a.G) {
        case 1: return launch_split_g<D, 1>(km, vm, a, grid, err, st);
        case 2: return launch_split_g<D, 2>(km, vm, a, grid, err, st);
        case 3: return launch_split_g<D, 3>(km, vm, a, grid, err, st);
        case 4: return launch_split_g<D, 4>(km, vm, a, grid, err, st);
        case 5: return launch_split_g<D, 5>(km, vm, a, grid, err, st);
        case 6: return launch_split_g<D, 6>(km, vm, a, grid, err, st);
        case 7: return launch_split_g<D, 7>(km, vm, a, grid, err, st);
        case 8: return launch_split_g<D, 8>(km, vm, a, grid, err, st);
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
    CUtensorMap km, vm;
    cudaError_t e = pool_maps(c, &km, &vm);
    if (e != cudaSuccess) return e;
    DecodeArgs a;
    a.layer = layer;
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
    e = c->head_dim == 128 ? launch_split<128>(km, vm, a, grid, err, st) : launch_split<64>(km, vm, a, grid, err, st);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.hq, (unsigned)n);
    cfg.blockDim = dim3((unsigned)c->head_dim);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return c->head_dim == 128 ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, a)
                              : cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, a);
}

size_t decode_workspace_bytes(const kara_cache *c, int32_t n, int32_t bt_stride)
{
    const size_t npart = (size_t)n * c->num_q_heads * decode_max_splits(bt_stride, c->block_size);
    return align256(npart * c->head_dim * sizeof(float)) + align256(npart * sizeof(float2));
}

}  // namespace kara
