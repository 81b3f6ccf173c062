"""Admission scheduler with periodic compression (host logic, CPU only).

The compressor is a host stand-in that applies the step's table rule -- new
length L' = L - C + R, fresh ids at [p0, p0 + n_new), -1 beyond, the old tail
[p0, ceil(L/bs)) freed -- so the scheduler's block accounting is checked
without a GPU.  The device path of the same rule is checked against the oracle
in the GPU tests."""
import math
import types

import pytest
import torch

from decode_kv_cache_03_gb300 import kara
from decode_kv_cache_03_gb300.periodic import AdmissionScheduler, BlockPool, PeriodicSchedule

BS = 16


class HostCompressor:
    def __init__(self, W, B, K, R):
        self.W, self.B, self.R = W, B, R
        self.params = kara.params(W, B, K, R, 0.1)
        self.k = types.SimpleNamespace(device=torch.device("cpu"))
        self.calls = 0

    def plan(self, lengths_host, bt_stride):
        return kara.kara_plan(self.params, BS, lengths_host, bt_stride)

    def compress(self, d_len, d_bt, q, fresh, freed, new_len, scores=None, cand=None, kept=None, stream=None):
        self.calls += 1
        fo = oo = 0
        for i in range(d_len.shape[0]):
            L = int(d_len[i])
            ws = L - self.W
            p0 = ws // BS
            n_old = math.ceil(L / BS) - p0
            Ln = ws + self.R + self.B
            n_new = math.ceil(Ln / BS) - p0
            freed[oo:oo + n_old] = d_bt[i, p0:p0 + n_old]
            d_bt[i, p0:p0 + n_new] = fresh[fo:fo + n_new]
            d_bt[i, p0 + n_new:p0 + n_old] = -1
            new_len[i] = Ln
            fo += n_new
            oo += n_old

    def error(self, stream=None):
        return 0


def check_accounting(sched, total):
    live = sched.live_blocks()
    free = sched.pool.free
    assert len(live) == len(set(live)) and len(free) == len(set(free))
    assert not set(live) & set(free)
    assert sorted(live + free) == list(range(total))
    for L, left, row in sched.running.values():
        assert len(row) == (L + BS - 1) // BS and left > 0
    assert sched.outstanding() <= len(free)      # every running sequence can finish


def simulate(compress, steps=1500, total=400, seed=0):
    rng = torch.Generator().manual_seed(seed)
    reqs = [(int(torch.randint(300, 400, (1,), generator=rng)), int(torch.randint(300, 900, (1,), generator=rng)))
            for _ in range(60)]
    sched = AdmissionScheduler(BlockPool(range(total)), reqs, BS, bt_stride=96)
    comp = HostCompressor(W=256, B=32, K=16, R=44)
    schedule = PeriodicSchedule(64, 0.5, 256, seed=seed)
    running = []
    for step in range(1, steps + 1):
        sched.admit()
        sched.step()
        if compress and schedule.due(step):
            sched.compress(comp, schedule, lambda n: None)
        check_accounting(sched, total)
        running.append(len(sched.running))
    return sched, running, comp


def test_accounting_without_compression():
    sched, running, _ = simulate(False)
    assert max(running) >= 2 and sched.finished
    # every decoded token is counted once: finished requests decoded all their
    # tokens, running ones what they have so far
    gen = {i: g for i, _, g in sched.requests}
    want = sum(gen[i] for i in sched.finished) + sum(gen[r] - left for r, (_, left, _) in sched.running.items())
    assert sched.tokens == want


def test_accounting_with_compression_and_more_concurrency():
    s0, r0, _ = simulate(False)
    s1, r1, comp = simulate(True)
    assert comp.calls > 0
    # compression frees blocks, so at least as many sequences run on average and more tokens decode
    assert sum(r1) > sum(r0)
    assert s1.tokens > s0.tokens


def test_admission_is_first_come_and_covers_whole_requests():
    # 20 blocks: request 0 needs ceil(300/16) = 19, request 1 needs 4 -> waits
    # although its prompt alone would fit; request 2 may not overtake it
    sched = AdmissionScheduler(BlockPool(range(20)), [(100, 200), (16, 40), (16, 1)], BS, bt_stride=20)
    assert sched.admit() == 1
    assert sorted(sched.running) == [0] and [w[0] for w in sched.waiting] == [1, 2]


def test_finished_sequences_return_their_blocks():
    sched = AdmissionScheduler(BlockPool(range(10)), [(15, 3)], BS, bt_stride=10)
    sched.admit()
    for _ in range(3):
        sched.step()
    assert sched.finished == [0] and not sched.running and sorted(sched.pool.free) == list(range(10))
    assert sched.tokens == 3
