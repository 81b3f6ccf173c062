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


class AdmissionScheduler:
    """Decoding sequences sharing a fixed pool of KV blocks, with optional
    periodic compression (summary, "Problem Statement" item 1 and section 3:
    memory bounds how many sequences decode at once, and the periodic policy
    frees blocks so more of them can).

    A request (prompt tokens, tokens to generate) waits in arrival order and is
    admitted when the pool can hold the blocks it will need to finish,
    counted from its current length without further compression, on top of
    what the running sequences may still need.  So no sequence ever waits for
    a block and the pool never deadlocks.  Each decode step appends one token to
    every running sequence; a sequence finishes once it has generated its
    tokens and returns its blocks.  With a compressor, every period of the
    schedule the chosen sequences go through compress_selected: their cached
    length drops by C - R, their freed blocks return to the pool, and the
    blocks they may still need shrink, so more requests are admitted.  No
    model runs: K/V contents are whatever the pool holds, and the window
    queries come from `q_window(n)`.
    """

    def __init__(self, pool: BlockPool, requests, block: int, bt_stride: int):
        self.pool, self.block, self.bt_stride = pool, block, bt_stride
        self.requests = [(i, int(p), int(g)) for i, (p, g) in enumerate(requests)]
        self.waiting = list(self.requests)
        self.running = {}          # request id -> [length, tokens left, table row (ids in logical order)]
        self.finished = []
        self.tokens = 0

    def _blocks(self, length: int) -> int:
        return (length + self.block - 1) // self.block

    def outstanding(self) -> int:
        """Blocks the running sequences may still take, without compression."""
        return sum(self._blocks(L + left) - len(row) for L, left, row in self.running.values())

    def admit(self) -> int:
        n = 0
        spare = len(self.pool.free) - self.outstanding()
        while self.waiting:
            rid, prompt, gen = self.waiting[0]
            need = self._blocks(prompt + gen)
            if need > spare or need > self.bt_stride:
                break
            self.waiting.pop(0)
            self.running[rid] = [prompt, gen, self.pool.take(self._blocks(prompt))]
            spare -= need
            n += 1
        return n

    def step(self) -> int:
        """One decode step; returns the tokens decoded."""
        done = []
        for rid, st in self.running.items():
            L, left, row = st
            if L % self.block == 0:
                row.append(self.pool.take(1)[0])
            st[0], st[1] = L + 1, left - 1
            if st[1] == 0:
                done.append(rid)
        for rid in done:
            self.pool.give(self.running.pop(rid)[2])
            self.finished.append(rid)
        decoded = len(self.running) + len(done)
        self.tokens += decoded
        return decoded

    def compress(self, comp, schedule: PeriodicSchedule, q_window) -> int:
        """Compress the schedule's choice among the running sequences; returns
        the blocks freed."""
        ids = sorted(self.running)
        if not ids:
            return 0
        lengths = [self.running[r][0] for r in ids]
        pick = schedule.choose(lengths)
        # fresh blocks leave the pool before the old ones come back: keep the
        # longest prefix of the choice the spare blocks can cover
        if pick:
            nn = comp.plan(torch.tensor([lengths[i] for i in pick], dtype=torch.int32), self.bt_stride)[0]
            spare = len(self.pool.free) - self.outstanding()
            keep, need = [], 0
            for j, i in enumerate(pick):
                need += int(nn[j])
                if need > spare:
                    break
                keep.append(i)
            pick = keep
        if not pick:
            return 0
        table = torch.full((len(ids), self.bt_stride), -1, dtype=torch.int32)
        for i, r in enumerate(ids):
            row = self.running[r][2]
            table[i, :len(row)] = torch.tensor(row, dtype=torch.int32)
        freed, status = compress_selected(comp, pick, lengths, table, q_window(len(pick)), self.pool)
        if status != 0:
            raise RuntimeError(f"compression failed: {kara.status_string(status)}")
        for i in pick:
            r = ids[i]
            L = int(lengths[i])
            self.running[r][0] = L
            self.running[r][2] = [int(x) for x in table[i, :self._blocks(L)]]
        return len(freed)

    def live_blocks(self) -> list[int]:
        return [b for st in self.running.values() for b in st[2]]
