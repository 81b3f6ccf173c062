"""Host-side driver of the periodic compression policy.

Follows the gist.science summary of Kara (arXiv 2607.01237), section "3. KvLLM
Framework and Periodic Compression": every fixed number of decode steps the
trailing blocks of selected sequences are compressed, which frees memory for
more concurrent sequences.  This module is the bookkeeping around the library
call: a pool of free physical blocks, block allocation as decoding appends
tokens, the choice of sequences at each period, and the hand-over of fresh ids
to, and freed ids back from, kara_compress_batch.  All device work stays in the
library; tables and lengths are mirrored on the host, as a scheduler keeps them.
"""
from __future__ import annotations

import math
import random

import torch

from . import kara


class BlockPool:
    """Free physical block ids.  `pinned` ids (shared blocks) are never recycled."""

    def __init__(self, free_ids, pinned=()):
        self.free = list(int(i) for i in free_ids)
        self.pinned = set(int(i) for i in pinned)

    def take(self, n: int) -> list[int]:
        if n > len(self.free):
            raise RuntimeError(f"block pool exhausted: need {n}, have {len(self.free)}")
        out, self.free = self.free[:n], self.free[n:]
        return out

    def give(self, ids) -> int:
        back = [int(i) for i in ids if int(i) not in self.pinned]
        self.free.extend(back)
        return len(back)


class PeriodicSchedule:
    """Every `interval` decode steps, a seeded random `fraction` of the eligible
    sequences (cached length >= W) is compressed."""

    def __init__(self, interval: int, fraction: float, W: int, seed: int = 0):
        self.interval, self.fraction, self.W = interval, fraction, W
        self.rng = random.Random(seed)

    def due(self, step: int) -> bool:
        return step > 0 and step % self.interval == 0

    def choose(self, lengths_host) -> list[int]:
        eligible = [s for s, L in enumerate(lengths_host) if int(L) >= self.W]
        m = min(len(eligible), math.ceil(self.fraction * len(lengths_host)))
        return sorted(self.rng.sample(eligible, m))


def append_tokens(lengths_host, table_host, pool: BlockPool, block: int) -> list[tuple[int, int, int]]:
    """One decode step: every sequence grows by one token.  Returns the
    (sequence, logical block, physical id) of blocks opened by this step."""
    opened = []
    for s in range(len(lengths_host)):
        L = int(lengths_host[s])
        if L % block == 0:
            bid = pool.take(1)[0]
            table_host[s, L // block] = bid
            opened.append((s, L // block, bid))
        lengths_host[s] = L + 1
    return opened


def compress_selected(comp, seqs, lengths_host, table_host, q_window, pool: BlockPool, stream=None, events=None,
                      scores=None, kept=None):
    """Compress the trailing windows of `seqs` with kara_compress_batch.

    comp: a Compressor; q_window: device bf16 [len(seqs)][layers][Hq][W][D].
    Updates lengths_host / table_host in place and returns
    (freed ids, device status).  events: optional (start, end) CUDA events
    recorded around the library call only; scores / kept: optional device
    outputs [len(seqs)][layers][Hkv][C] / [..][R]."""
    dev = comp.k.device
    sel_len = torch.tensor([int(lengths_host[s]) for s in seqs], dtype=torch.int32)
    sel_bt = table_host[seqs].contiguous()
    nn, no, tn, to = comp.plan(sel_len, sel_bt.shape[1])
    fresh = torch.tensor(pool.take(tn), dtype=torch.int32, device=dev)
    d_len = sel_len.to(dev)
    d_bt = sel_bt.to(dev)
    freed = torch.empty(max(to, 1), dtype=torch.int32, device=dev)
    new_len = torch.empty(len(seqs), dtype=torch.int32, device=dev)
    if events:
        events[0].record()
    comp.compress(d_len, d_bt, q_window, fresh, freed, new_len, scores=scores, kept=kept, stream=stream)
    if events:
        events[1].record()
    status = comp.error(stream)
    if status != 0:
        pool.give(fresh.tolist())
        return [], status
    table_host[seqs] = d_bt.cpu()
    nl = new_len.cpu()
    for i, s in enumerate(seqs):
        lengths_host[s] = int(nl[i])
    fr = freed[:to].cpu().tolist()
    pool.give(fr)
    return fr, status
