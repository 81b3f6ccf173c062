"""Pins for the oracle's compaction of the window-query ring (CPU only).

The ring holds the query of logical position x in row x mod W.  The pins
compare against the logical (position-ordered) view of the same queries, so a
wrong modulus, a wrong source row or a missed buffer row fails; they also tie
the moved queries to the K rows the K/V compaction moves to the same place,
and check that the window scores do not depend on the ring's rotation."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import random_spec


def make_ring(wl, rng):
    """Window queries in logical order q_log [n][l][h][W][d] and the ring that
    holds them (row (ws + i) mod W = logical row i), as uint16 bits."""
    sp = wl.spec
    q_log = wl.q.view(torch.int16).numpy().view(np.uint16).copy()
    ring = np.empty_like(q_log)
    for s in range(sp.n_seq):
        ws = int(wl.lengths[s]) - sp.W
        rows = (ws + np.arange(sp.W)) % sp.W
        ring[s][:, :, rows] = q_log[s]
    return q_log, ring


def random_kept(sp, rng):
    C = sp.W - sp.B
    return np.stack([np.sort(rng.choice(C, sp.R, replace=False)) for _ in range(sp.n_seq * sp.layers * sp.hkv)]
                    ).reshape(sp.n_seq, sp.layers, sp.hkv, sp.R).astype(np.int32)


@pytest.mark.parametrize("seed,G,W,B,R", [(81, 2, 64, 16, 20), (82, 1, 48, 8, 39), (83, 3, 64, 0, 5)])
def test_kept_and_buffer_queries_land_at_their_new_positions(seed, G, W, B, R):
    sp = random_spec(seed, G=G, W=W, B=B, D=32, len_lo=W, len_hi=W + 90, R=R)
    wl = synth.generate(sp)
    rng = np.random.default_rng(seed)
    q_log, ring = make_ring(wl, rng)
    kept = random_kept(sp, rng)
    new = oracle.compact_queries(oracle.shape_of(wl), ring, wl.lengths, kept)
    for s in range(sp.n_seq):
        ws = int(wl.lengths[s]) - W
        for l in range(sp.layers):
            for h in range(sp.hq):
                src = np.concatenate([kept[s, l, h // G], np.arange(W - B, W)])     # logical window rows
                dst = (ws + np.arange(R + B)) % W                                 # ring rows of ws .. ws+R+B-1
                np.testing.assert_array_equal(new[s, l, h, dst], q_log[s, l, h, src])
                rest = (ws + np.arange(R + B, W)) % W                             # rows of positions past L'
                np.testing.assert_array_equal(new[s, l, h, rest], ring[s, l, h, rest])


def test_queries_follow_their_keys():
    """After both compactions, new position x holds the query and the key of the
    same old position, for every kept and buffer row."""
    sp = random_spec(84, G=2, W=64, B=16, D=32, len_lo=100, len_hi=200, K=6, R=20)
    wl = synth.generate(sp)
    rng = np.random.default_rng(84)
    q_log, ring = make_ring(wl, rng)
    kept = random_kept(sp, rng)
    kh = wl.k.view(torch.int16).numpy().view(np.uint16)
    vh = wl.v.view(torch.int16).numpy().view(np.uint16)
    st, k2, _, bt2, _, _ = oracle.compact(oracle.shape_of(wl), kh, vh, wl.block_table, wl.lengths, kept, wl.fresh)
    assert st == oracle.OK
    newq = oracle.compact_queries(oracle.shape_of(wl), ring, wl.lengths, kept)
    bt = wl.block_table.numpy()
    for s in range(sp.n_seq):
        L = int(wl.lengths[s])
        ws = L - sp.W
        for r, x_old in enumerate(np.concatenate([ws + kept[s, 1, 0], np.arange(L - sp.B, L)])):
            x_new = ws + r
            k_new = k2[1, bt2[s, x_new // 16], 0, x_new % 16]
            k_old = kh[1, bt[s, x_old // 16], 0, x_old % 16]
            np.testing.assert_array_equal(k_new, k_old)
            for h in range(2):        # query heads of KV head 0
                np.testing.assert_array_equal(newq[s, 1, h, x_new % sp.W], q_log[s, 1, h, x_old - ws])


def test_full_budget_is_the_identity():
    sp = random_spec(85, G=2, W=64, B=16, D=32, len_lo=70, len_hi=130, R=48)
    wl = synth.generate(sp)
    _, ring = make_ring(wl, np.random.default_rng(0))
    kept = np.broadcast_to(np.arange(48, dtype=np.int32), (sp.n_seq, sp.layers, sp.hkv, 48)).copy()
    new = oracle.compact_queries(oracle.shape_of(wl), ring, wl.lengths, kept)
    np.testing.assert_array_equal(new, ring)


def test_scores_do_not_depend_on_the_rotation():
    """The softmax of each query row and the sum over rows do not see the rows'
    order, so the ring scores like the linear window."""
    sp = random_spec(86, G=2, W=64, B=16, D=32, len_lo=70, len_hi=150)
    wl = synth.generate(sp)
    _, ring = make_ring(wl, np.random.default_rng(1))
    _, c_lin = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths, with_colsum=True)
    _, c_ring = oracle.scores(oracle.shape_of(wl), torch.from_numpy(ring.view(np.int16)), wl.k, wl.block_table,
                              wl.lengths, with_colsum=True)
    np.testing.assert_allclose(c_ring, c_lin, rtol=1e-12)
