"""Seeded synthetic workloads for the decode-time KV-cache compression step.

This module only draws inputs: window queries, a paged bf16 K/V pool, cached
lengths, block tables and a list of fresh block ids, with the shapes and value
structure of the five model-shaped workloads (planted key directions, planted
spans, heavy-tailed keys, ragged lengths, shuffled physical blocks).  It holds
none of the compression method's arithmetic: no scores, no selection, no page
plan.  Both the CUDA path's tests and the CPU oracle's tests take their inputs
from here, so neither side generates data for the other.

Layouts (all row-major, D contiguous):
  q      bf16 [n_seq][layers][hq][W][d]          window queries
  k, v   bf16 [layers][num_blocks][hkv][block][d] paged pools
  lengths int32 [n_seq]                           cached tokens per sequence
  block_table int32 [n_seq][bt_stride]            logical block -> physical id
  fresh  int32 [n_fresh]                          unused physical ids

Pool regions (physical ids, in this order):
  [0, P)           shared prefix pool (only with alias_prefix): logical blocks
                   far before the trailing window of every sequence alias
                   these few blocks; a window never reaches them.
  [P, P + Nd)      distinct blocks owned by one sequence each.
  [P + Nd, ...)    fresh blocks, filled with a canary pattern.
"""
from __future__ import annotations

import dataclasses
import math

import torch

CANARY_BF16_BITS = 0x7FA5  # a quiet-NaN bf16 pattern no generator draw produces


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    n_seq: int
    layers: int
    hq: int
    hkv: int
    d: int
    block: int
    W: int
    B: int
    K: int
    R: int
    lam: float
    len_lo: int
    len_hi: int          # inclusive
    shuffled: bool
    plant: str           # 'count' | 'bernoulli' | 'spans' | 'heavy' | 'none'
    plant_arg: float
    seed: int

    @property
    def C(self) -> int:
        return self.W - self.B

    @property
    def G(self) -> int:
        return self.hq // self.hkv

    @property
    def n_windows(self) -> int:
        return self.n_seq * self.layers * self.hkv

    def with_(self, **kw) -> "Spec":
        return dataclasses.replace(self, **kw)


def _budget(pct: int, W: int, B: int) -> int:
    """Retained-token budget given as a percentage of the compressible region."""
    return (pct * (W - B)) // 100


SPECS: dict[str, Spec] = {
    # 1 sequence, 1 layer, 4 q / 2 kv heads, d 64, 256 cached tokens; W 64 = 48 + 16.
    "tiny": Spec("tiny", 1, 1, 4, 2, 64, 16, 64, 16, 8, 16, 0.1, 256, 256,
                 False, "count", 4, 0),
    # Qwen3-4B shape: 36 layers, 32/8 heads, d 128; 32 x 4096 tokens, shuffled ids.
    "qwen3_4b": Spec("qwen3_4b", 32, 36, 32, 8, 128, 16, 512, 64, 64, _budget(20, 512, 64),
                     0.1, 4096, 4096, True, "bernoulli", 0.05, 1),
    # Qwen3-14B shape: 40 layers, 40/8 heads, d 128; 128 sequences of 2048..16384.
    "qwen3_14b": Spec("qwen3_14b", 128, 40, 40, 8, 128, 16, 1024, 128, 128,
                      _budget(30, 1024, 128), 0.1, 2048, 16384, False, "spans", 0.08, 2),
    # Llama-8B shape: 32 layers, 32/8 heads, d 128; 64 sequences of 1024..8192, shuffled.
    "llama_8b": Spec("llama_8b", 64, 32, 32, 8, 128, 16, 256, 32, 32, _budget(10, 256, 32),
                     0.1, 1024, 8192, True, "heavy", 0.01, 3),
}


def sweep_spec(batch: int, W: int, index: int = 0) -> Spec:
    """Periodic-policy sweep point on the Qwen3-4B shape: buffer W/8, Top-K W/8, 20 %."""
    B = W // 8
    return Spec(f"sweep_b{batch}_w{W}", batch, 36, 32, 8, 128, 16, W, B, max(1, W // 8),
                _budget(20, W, B), 0.1, 4096, 4096, True, "bernoulli", 0.05, 4 + index)


@dataclasses.dataclass
class Workload:
    spec: Spec
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    lengths: torch.Tensor
    block_table: torch.Tensor
    fresh: torch.Tensor
    prefix_pool: int          # P: ids [0, P) are the shared prefix pool
    fresh_base: int           # first fresh physical id

    @property
    def num_blocks(self) -> int:
        return self.k.shape[1]

    @property
    def bt_stride(self) -> int:
        return self.block_table.shape[1]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _unit_dirs(layers: int, hkv: int, d: int, gen, device) -> torch.Tensor:
    u = torch.randn(layers, hkv, d, generator=gen, device=device, dtype=torch.float32)
    return u / u.norm(dim=-1, keepdim=True)


def _plant_mask(spec: Spec, gen, device) -> torch.Tensor:
    """[layers][hkv][W] float mask of planted window positions (window-relative)."""
    L, H, W, C = spec.layers, spec.hkv, spec.W, spec.C
    m = torch.zeros(L, H, W, device=device, dtype=torch.float32)
    if spec.plant == "count":
        n = int(spec.plant_arg)
        for li in range(L):
            for h in range(H):
                pos = torch.randperm(C, generator=gen, device=device)[:n]
                m[li, h, pos] = 1.0
    elif spec.plant == "bernoulli":
        r = torch.rand(L, H, C, generator=gen, device=device)
        m[:, :, :C] = (r < spec.plant_arg).float()
    elif spec.plant == "spans":
        target = int(round(spec.plant_arg * W))
        host = torch.zeros(L, H, W, dtype=torch.float32)
        cpu_gen = torch.Generator().manual_seed(
            int(torch.randint(0, 2**31 - 1, (1,), generator=gen, device=device).item()))
        for li in range(L):
            for h in range(H):
                lens, total = [], 0
                while total < target:
                    ln = int(torch.randint(2, 33, (1,), generator=cpu_gen).item())
                    ln = min(ln, target - total)
                    lens.append(ln)
                    total += ln
                free = C - total
                # random non-overlapping placement: gaps from sorted cut points
                cuts = torch.sort(torch.randint(0, free + 1, (len(lens),), generator=cpu_gen)).values
                pos = 0
                prev = 0
                for ln, c in zip(lens, cuts.tolist()):
                    pos += c - prev
                    prev = c
                    host[li, h, pos:pos + ln] = 1.0
                    pos += ln
        m = host.to(device)
    return m


def generate(spec: Spec, device="cpu", alias_prefix: bool | None = None,
             prefix_pool_blocks: int = 16, with_q: bool = True, extra_fresh_per_seq: int = 0,
             fresh_per_seq: int | None = None) -> Workload:
    """Draw one workload.  Deterministic for a given (spec, device type).

    with_q=False leaves q as None (a caller that draws query windows itself);
    fresh_per_seq sets the pool of unused blocks per sequence (default: a
    window's worth, W/16 + 1) and extra_fresh_per_seq adds to it."""
    dev = torch.device(device)
    gen = _gen(spec.seed, dev)
    n, Lyr, Hq, Hk, D, bs, W = (spec.n_seq, spec.layers, spec.hq, spec.hkv, spec.d,
                                 spec.block, spec.W)
    G = Hq // Hk
    if alias_prefix is None:
        alias_prefix = dev.type == "cuda"

    # cached lengths
    if spec.len_lo == spec.len_hi:
        lengths = torch.full((n,), spec.len_lo, dtype=torch.int32)
    else:
        lengths = torch.randint(spec.len_lo, spec.len_hi + 1, (n,), generator=_gen(spec.seed + 1000, "cpu"),
                                dtype=torch.int64).to(torch.int32)
    nblk_seq = [(int(l) + bs - 1) // bs for l in lengths]
    bt_stride = max(nblk_seq)
    tail = W // bs + 1      # trailing logical blocks that get distinct storage when aliasing

    # physical ids
    P = prefix_pool_blocks if alias_prefix else 0
    distinct_counts = [min(nb, tail) if alias_prefix else nb for nb in nblk_seq]
    Nd = sum(distinct_counts)
    per_seq_fresh = (W // bs + 1 if fresh_per_seq is None else fresh_per_seq) + extra_fresh_per_seq
    n_fresh = n * per_seq_fresh
    num_blocks = P + Nd + n_fresh
    host_gen = _gen(spec.seed + 2000, "cpu")
    dist_ids = torch.arange(P, P + Nd, dtype=torch.int32)
    fresh_ids = torch.arange(P + Nd, P + Nd + n_fresh, dtype=torch.int32)
    if spec.shuffled:
        dist_ids = dist_ids[torch.randperm(Nd, generator=host_gen)]
        fresh_ids = fresh_ids[torch.randperm(n_fresh, generator=host_gen)]
    bt = torch.full((n, bt_stride), -1, dtype=torch.int32)
    off = 0
    for s in range(n):
        nb, nd = nblk_seq[s], distinct_counts[s]
        for t in range(nb - nd):
            bt[s, t] = (s * 7 + t) % P
        bt[s, nb - nd:nb] = dist_ids[off:off + nd]
        off += nd

    # pools: N(0,1) bf16, fresh region = canary
    k = torch.empty(Lyr, num_blocks, Hk, bs, D, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    for li in range(Lyr):
        k[li].copy_(torch.randn(num_blocks, Hk, bs, D, generator=gen, device=dev))
        v[li].copy_(torch.randn(num_blocks, Hk, bs, D, generator=gen, device=dev))
    canary = torch.tensor([CANARY_BF16_BITS], dtype=torch.int16).view(torch.bfloat16).to(dev)
    k[:, P + Nd:].copy_(canary.expand_as(k[:, P + Nd:]))
    v[:, P + Nd:].copy_(canary.expand_as(v[:, P + Nd:]))

    # window keys with structure, written through the block table
    u = _unit_dirs(Lyr, Hk, D, gen, dev)
    q = torch.empty(n, Lyr, Hq, W, D, dtype=torch.bfloat16, device=dev) if with_q else None
    bt_dev = bt.to(dev)
    planted_q = spec.plant in ("count", "bernoulli", "spans")
    for s in range(n):
        Ls = int(lengths[s])
        # a sequence shorter than the window (decode-only workloads) holds only
        # the window's last Ls positions; the draws below stay a full window's
        first = max(W - Ls, 0)
        pos = torch.arange(Ls - W + first, Ls, device=dev)
        blk = bt_dev[s, pos // bs].long()
        slot = pos % bs
        kw = torch.randn(Lyr, Hk, W, D, generator=gen, device=dev)
        if spec.plant == "heavy":
            r = torch.rand(Lyr, Hk, W, generator=gen, device=dev)
            sign = torch.where(torch.rand(Lyr, Hk, W, generator=gen, device=dev) < 0.5, -1.0, 1.0)
            scale = torch.where(r < spec.plant_arg, 4.0 * sign, torch.ones_like(sign))
            kw = kw * scale[..., None]
        elif spec.plant != "none":
            m = _plant_mask(spec, gen, dev)
            kw = kw + 3.0 * m[..., None] * u[:, :, None, :]
        k[:, blk, :, slot, :] = kw[:, :, first:].permute(2, 0, 1, 3).to(torch.bfloat16)
        if not with_q:
            continue
        qs = torch.randn(Lyr, Hq, W, D, generator=gen, device=dev)
        if planted_q:
            uq = u.repeat_interleave(G, dim=1)          # [layers][hq][D]
            qs = qs + 1.5 * uq[:, :, None, :]
        q[s].copy_(qs.to(torch.bfloat16))

    return Workload(spec, q, k, v, lengths.to(dev), bt_dev, fresh_ids.to(dev), P, P + Nd)


def host_subset(wl: Workload, seqs: list[int]) -> Workload:
    """Copy the data of a few sequences to host memory with compacted block ids.

    Every block the selected sequences' tables reference is copied; ids are
    renumbered densely in order of first appearance.  Fresh blocks for the
    subset are appended as new canary-filled blocks (one window's worth per
    sequence), so the subset is a self-contained workload.
    """
    spec = wl.spec.with_(n_seq=len(seqs))
    bt = wl.block_table[seqs].cpu()
    lengths = wl.lengths[seqs].cpu()
    ids = []
    seen = {}
    for s in range(len(seqs)):
        nb = (int(lengths[s]) + spec.block - 1) // spec.block
        for t in range(nb):
            b = int(bt[s, t])
            if b not in seen:
                seen[b] = len(ids)
                ids.append(b)
    remap = torch.full((wl.num_blocks,), -1, dtype=torch.int32)
    idx = torch.tensor(ids, dtype=torch.int64)
    remap[idx] = torch.arange(len(ids), dtype=torch.int32)
    new_bt = torch.where(bt >= 0, remap[bt.clamp(min=0).long()], torch.full_like(bt, -1))
    per_seq_fresh = spec.W // spec.block + 1
    n_fresh = len(seqs) * per_seq_fresh
    kk = wl.k[:, idx.to(wl.k.device)].cpu()
    vv = wl.v[:, idx.to(wl.v.device)].cpu()
    canary = torch.tensor([CANARY_BF16_BITS], dtype=torch.int16).view(torch.bfloat16)
    pad = canary.expand(spec.layers, n_fresh, spec.hkv, spec.block, spec.d)
    k = torch.cat([kk, pad], dim=1).contiguous()
    v = torch.cat([vv, pad], dim=1).contiguous()
    fresh = torch.arange(len(ids), len(ids) + n_fresh, dtype=torch.int32)
    q = wl.q[seqs].cpu().contiguous()
    return Workload(spec, q, k, v, lengths.clone(), new_bt.contiguous(), fresh, 0, len(ids))


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """Raw 16-bit patterns of a bf16 tensor (as int16)."""
    return t.contiguous().view(torch.int16)


def decode_queries(spec: Spec, seed: int = 0, device="cpu") -> torch.Tensor:
    """One decode query per sequence and query head: bf16 [n_seq][hq][d], ~N(0,1)."""
    g = _gen(10_000 + seed, device)
    return torch.randn(spec.n_seq, spec.hq, spec.d, generator=g, device=device).to(torch.bfloat16)
