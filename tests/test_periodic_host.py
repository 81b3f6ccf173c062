"""Host bookkeeping of the periodic policy (CPU): block pool, schedule, decode appends.

Compressions are simulated with the host page plan (kara_plan): a compressed
sequence takes n_new fresh blocks and returns its n_old old tail blocks, as the
library does; the test checks that no block is ever lost or owned twice.
"""
import math

import numpy as np
import torch

from decode_kv_cache_03_gb300 import build

build.build()
from decode_kv_cache_03_gb300 import kara  # noqa: E402
from decode_kv_cache_03_gb300.periodic import BlockPool, PeriodicSchedule, append_tokens  # noqa: E402


def test_schedule_due_and_choice_are_deterministic():
    s1 = PeriodicSchedule(128, 0.5, 256, seed=3)
    s2 = PeriodicSchedule(128, 0.5, 256, seed=3)
    assert [t for t in range(600) if s1.due(t)] == [128, 256, 384, 512]
    lengths = [300, 100, 256, 900, 255, 1000, 4000, 12]
    a, b = s1.choose(lengths), s2.choose(lengths)
    assert a == b and len(a) == math.ceil(0.5 * len(lengths)) and all(lengths[i] >= 256 for i in a)
    assert PeriodicSchedule(1, 1.0, 5000).choose(lengths) == []


def test_pool_never_loses_or_duplicates_blocks():
    rng = np.random.default_rng(0)
    n, bs, W, B, R = 12, 16, 128, 16, 22
    lengths = rng.integers(W, 600, size=n).tolist()
    stride = 200
    table = torch.full((n, stride), -1, dtype=torch.int32)
    nid = 0
    for s in range(n):
        for t in range((lengths[s] + bs - 1) // bs):
            table[s, t] = nid
            nid += 1
    total = 4000
    pool = BlockPool(range(nid, total))
    sched = PeriodicSchedule(64, 0.5, W, seed=1)
    p = kara.params(W, B, 8, R, 0.1)
    for step in range(1, 300):
        append_tokens(lengths, table, pool, bs)
        if sched.due(step):
            seqs = sched.choose(lengths)
            sel_len = torch.tensor([lengths[s] for s in seqs], dtype=torch.int32)
            nn, no, tn, to = kara.kara_plan(p, bs, sel_len, stride)
            fresh = pool.take(tn)
            off = 0
            for i, s in enumerate(seqs):
                L = lengths[s]
                p0 = (L - W) // bs
                old = table[s, p0:p0 + int(no[i])].tolist()
                table[s, p0:p0 + int(no[i])] = -1
                table[s, p0:p0 + int(nn[i])] = torch.tensor(fresh[off:off + int(nn[i])], dtype=torch.int32)
                off += int(nn[i])
                lengths[s] = L - (W - B) + R
                pool.give(old)
        live = [int(x) for s in range(n) for x in table[s, :(lengths[s] + bs - 1) // bs].tolist()]
        assert len(live) == len(set(live)) and -1 not in live
        assert not (set(live) & set(pool.free))
        assert len(live) + len(pool.free) == total
    assert max(lengths) < stride * bs


def test_pinned_blocks_are_not_recycled():
    pool = BlockPool([10, 11], pinned=[1, 2])
    assert pool.give([1, 5, 2, 6]) == 2
    assert pool.free == [10, 11, 5, 6]
