"""Pins for the oracle's page plan and gather-compaction (CPU only)."""
import numpy as np
import pytest

import oracle
import synth
from _cases import random_spec


def blocks_covering(lo, hi, bs):
    """Logical blocks touched by positions [lo, hi), by enumeration."""
    return sorted({x // bs for x in range(lo, hi)})


@pytest.mark.parametrize("seed", range(8))
def test_plan_counts_by_enumeration(seed):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([4, 8, 16]))
    W = int(rng.integers(2, 80))
    B = int(rng.integers(0, W))
    R = int(rng.integers(1, W - B + 1))
    lengths = rng.integers(W, W + 200, size=12).astype(np.int32)
    bt_stride = int((lengths.max() + bs - 1) // bs)
    nn, no = oracle.plan(lengths, W, B, R, bs, bt_stride)
    for L, a, b in zip(lengths.tolist(), nn.tolist(), no.tolist()):
        ws = L - W
        first = ws // bs
        old = [t for t in blocks_covering(0, L, bs) if t >= first]
        new_len = L - (W - B) + R
        new = [t for t in blocks_covering(0, new_len, bs) if t >= first]
        assert (a, b) == (len(new), len(old))
        assert a <= b


def test_plan_rejects():
    with pytest.raises(ValueError):
        oracle.plan(np.int32([10]), 16, 4, 3, 16, 4)            # L < W
    with pytest.raises(ValueError):
        oracle.plan(np.int32([100]), 16, 4, 3, 16, 4)           # table too short
    with pytest.raises(ValueError):
        oracle.plan(np.int32([100]), 16, 4, 13, 16, 16)         # R > C


def run_compact(wl, seed=0):
    s = wl.spec
    rng = np.random.default_rng(seed)
    kept = np.zeros((s.n_seq, s.layers, s.hkv, s.R), np.int32)
    for idx in np.ndindex(s.n_seq, s.layers, s.hkv):
        kept[idx] = np.sort(rng.choice(s.C, size=s.R, replace=False))
    st, k2, v2, bt2, freed, new_len = oracle.compact(oracle.shape_of(wl), wl.k, wl.v, wl.block_table,
                                                     wl.lengths, kept, wl.fresh)
    assert st == oracle.OK
    return kept, k2, v2, bt2, freed, new_len


@pytest.mark.parametrize("seed,shuffled,block", [(1, True, 16), (2, False, 16), (3, True, 8), (4, True, 4)])
def test_compaction_moves_exact_rows(seed, shuffled, block):
    spec = random_spec(seed, G=2, hkv=2, W=64, B=16, D=32, block=block, n_seq=3, layers=2,
                       shuffled=shuffled, R=20)
    wl = synth.generate(spec)
    kept, k2, v2, bt2, freed, new_len = run_compact(wl, seed)
    k0 = wl.k.view(-1).view(__import__("torch").int16).numpy().view(np.uint16).reshape(wl.k.shape)
    v0 = wl.v.view(-1).view(__import__("torch").int16).numpy().view(np.uint16).reshape(wl.v.shape)
    bt0 = wl.block_table.numpy()
    bs, W, B, R = spec.block, spec.W, spec.B, spec.R
    for s_ in range(spec.n_seq):
        L = int(wl.lengths[s_])
        ws = L - W
        assert new_len[s_] == L - (W - B) + R
        # the new logical sequence of the window region, listed independently
        for li in range(spec.layers):
            for g in range(spec.hkv):
                src_pos = list(range((ws // bs) * bs, ws)) + [ws + int(j) for j in kept[s_, li, g]] \
                    + list(range(L - B, L))
                for n_i, xo in enumerate(src_pos):
                    xn = (ws // bs) * bs + n_i
                    ob, os_ = bt0[s_, xo // bs], xo % bs
                    nb, ns = bt2[s_, xn // bs], xn % bs
                    assert np.array_equal(k2[li, nb, g, ns], k0[li, ob, g, os_])
                    assert np.array_equal(v2[li, nb, g, ns], v0[li, ob, g, os_])
        # untouched prefix of the table
        first = ws // bs
        assert np.array_equal(bt2[s_, :first], bt0[s_, :first])
        nb_new = (int(new_len[s_]) + bs - 1) // bs
        nb_old = (L + bs - 1) // bs
        assert np.all(bt2[s_, nb_new:nb_old] == -1)
        assert np.array_equal(bt2[s_, nb_old:], bt0[s_, nb_old:])


@pytest.mark.parametrize("seed", [5, 6])
def test_compaction_touches_only_fresh_blocks(seed):
    spec = random_spec(seed, G=2, hkv=2, W=64, B=16, D=32, n_seq=4, layers=2, R=12)
    wl = synth.generate(spec)
    kept, k2, v2, bt2, freed, new_len = run_compact(wl, seed)
    import torch
    k0 = wl.k.view(torch.int16).numpy().view(np.uint16)
    v0 = wl.v.view(torch.int16).numpy().view(np.uint16)
    fresh = set(wl.fresh.tolist())
    changed = {b for b in range(wl.num_blocks)
               if not (np.array_equal(k2[:, b], k0[:, b]) and np.array_equal(v2[:, b], v0[:, b]))}
    assert changed <= fresh
    # freed + live = old live set, disjoint; fresh ids used are live now
    old_live = set()
    new_live = set()
    for s_ in range(spec.n_seq):
        nb_old = (int(wl.lengths[s_]) + spec.block - 1) // spec.block
        nb_new = (int(new_len[s_]) + spec.block - 1) // spec.block
        old_live |= set(wl.block_table[s_, :nb_old].tolist())
        new_live |= set(bt2[s_, :nb_new].tolist())
    fr = set(freed.tolist())
    assert len(fr) == len(freed)
    assert fr | (new_live - fresh) == old_live and not (fr & new_live)
    # slots past the new length in the last fresh block keep the canary
    for s_ in range(spec.n_seq):
        Lp = int(new_len[s_])
        if Lp % spec.block:
            b = bt2[s_, Lp // spec.block]
            assert np.all(k2[:, b, :, Lp % spec.block:] == synth.CANARY_BF16_BITS)


def test_compaction_rejects_short_fresh_list_and_bad_kept():
    spec = random_spec(7, W=64, B=16, D=32, n_seq=2, layers=1, R=10)
    wl = synth.generate(spec)
    kept = np.tile(np.arange(10, dtype=np.int32), (2, 1, spec.hkv, 1))
    st = oracle.compact(oracle.shape_of(wl), wl.k, wl.v, wl.block_table, wl.lengths, kept, wl.fresh[:1])[0]
    assert st == oracle.ENOBLOCKS
    bad = kept.copy()
    bad[0, 0, 0, 0] = spec.C
    st = oracle.compact(oracle.shape_of(wl), wl.k, wl.v, wl.block_table, wl.lengths, bad, wl.fresh)[0]
    assert st == oracle.EINVAL
    bt = wl.block_table.clone()
    L = int(wl.lengths[0])
    bt[0, (L - 1) // spec.block] = wl.num_blocks + 5
    st = oracle.compact(oracle.shape_of(wl), wl.k, wl.v, bt, wl.lengths, kept, wl.fresh)[0]
    assert st == oracle.EBADBLOCK


def test_compaction_rejects_repeated_or_live_fresh_ids():
    """A fresh id the plan consumes must be new: not an earlier fresh id, not any
    block the batch's tables still list (prefix blocks kept, tail blocks read)."""
    spec = random_spec(17, W=64, B=16, D=32, n_seq=3, layers=1, R=10, len_lo=100, len_hi=180)
    wl = synth.generate(spec)
    sh = oracle.shape_of(wl)
    kept = np.tile(np.arange(10, dtype=np.int32), (3, 1, spec.hkv, 1))
    nn, _ = oracle.plan(wl.lengths, spec.W, spec.B, spec.R, spec.block, wl.bt_stride)
    used = int(nn.sum())
    assert oracle.compact(sh, wl.k, wl.v, wl.block_table, wl.lengths, kept, wl.fresh)[0] == oracle.OK

    def status(fresh):
        return oracle.compact(sh, wl.k, wl.v, wl.block_table, wl.lengths, kept, fresh)[0]

    f = wl.fresh.clone()
    f[used - 1] = f[0]                                   # repeated within the consumed prefix
    assert status(f) == oracle.EDUPBLOCK
    f = wl.fresh.clone()
    f[1] = wl.block_table[2, 0]                          # a prefix block another sequence keeps
    assert status(f) == oracle.EDUPBLOCK
    L1 = int(wl.lengths[1])
    f = wl.fresh.clone()
    f[0] = wl.block_table[1, (L1 - 1) // spec.block]     # an old tail block the step reads
    assert status(f) == oracle.EDUPBLOCK
    f = wl.fresh.clone()
    f[used:] = f[0]                                      # ids past the consumed prefix are never used
    assert status(f) == oracle.OK


def test_compaction_rejects_unsorted_or_repeated_kept():
    spec = random_spec(18, W=64, B=16, D=32, n_seq=2, layers=1, R=10)
    wl = synth.generate(spec)
    sh = oracle.shape_of(wl)
    kept = np.tile(np.arange(10, dtype=np.int32), (2, 1, spec.hkv, 1))
    for mutate in (lambda k: k.__setitem__((1, 0, 1, 3), 1),            # repeats position 1
                   lambda k: k.__setitem__((0, 0, 0, slice(4, 6)), [5, 4])):  # out of order
        bad = kept.copy()
        mutate(bad)
        assert oracle.compact(sh, wl.k, wl.v, wl.block_table, wl.lengths, bad, wl.fresh)[0] == oracle.EINVAL
