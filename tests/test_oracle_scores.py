"""Pins for the oracle's window scores (CPU only).

Each check is chosen so that a plausible slip in the oracle -- a wrong scale,
a softmax over the wrong keys, a transposed operand, a dropped head, a wrong
block or slot in the addressing -- fails at least one of them.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import golden_case, independent_colsum, load_golden, random_spec


@pytest.mark.parametrize("name", ["score_hand.json", "address_hand.json"])
def test_hand_worked_fixtures(name):
    g = load_golden(name)
    shape, q, kpool, bt, ln = golden_case(g)
    s, cs = oracle.scores(shape, q, kpool, bt, ln, with_colsum=True)
    np.testing.assert_allclose(cs.reshape(-1), g["expected_colsum"], rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(s.reshape(-1), np.asarray(g["expected_scores"], np.float32))


@pytest.mark.parametrize("seed,G,W,B,D,block", [
    (11, 1, 64, 16, 64, 16), (12, 2, 64, 8, 64, 16), (13, 4, 32, 4, 32, 8), (14, 3, 48, 16, 16, 16),
    (15, 2, 128, 16, 128, 16)])
def test_matches_independent_fp64_softmax(seed, G, W, B, D, block):
    """Library softmax (torch fp64) over a numpy gather through the block table."""
    spec = random_spec(seed, G=G, W=W, B=B, D=D, block=block)
    wl = synth.generate(spec)
    s, cs = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths, with_colsum=True)
    ref = independent_colsum(wl)
    np.testing.assert_allclose(cs, ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(s, ref[..., :spec.C].astype(np.float32), rtol=2 ** -23, atol=0)


@pytest.mark.parametrize("seed", [21, 22, 23])
def test_row_sums(seed):
    """Every softmax row sums to one: sum_{j<W} t[j] = G*W; compressible part <= G*W."""
    spec = random_spec(seed, G=3, W=64, B=24, D=32, block=16, plant="bernoulli")
    wl = synth.generate(spec)
    s, cs = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths, with_colsum=True)
    G = spec.hq // spec.hkv
    np.testing.assert_allclose(cs.sum(-1), G * spec.W, rtol=1e-12)
    assert np.all(s.astype(np.float64).sum(-1) <= G * spec.W * (1 + 1e-6))
    assert np.all(s > 0)


def test_zero_queries_give_G_everywhere():
    spec = random_spec(31, G=4, W=64, B=16, D=64)
    wl = synth.generate(spec)
    wl.q.zero_()
    s = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths)
    np.testing.assert_array_equal(s, np.full_like(s, 4.0))


def test_equal_keys_give_G_everywhere():
    spec = random_spec(32, G=2, W=64, B=16, D=64, shuffled=False)
    wl = synth.generate(spec)
    row = torch.randn(spec.d).to(torch.bfloat16)
    wl.k[:] = row                                     # every key identical
    s = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths)
    np.testing.assert_allclose(s, 2.0, rtol=1e-6)


def test_group_heads_are_summed():
    """G identical query heads give exactly G times the one-head score."""
    base = random_spec(33, G=1, hkv=2, W=64, B=16, D=64)
    wl1 = synth.generate(base)
    s1, c1 = oracle.scores(oracle.shape_of(wl1), wl1.q, wl1.k, wl1.block_table, wl1.lengths,
                           with_colsum=True)
    G = 3
    spec3 = base.with_(hq=G * base.hkv)
    q3 = wl1.q.repeat_interleave(G, dim=2).contiguous()
    sh3 = oracle.make_shape(spec3.n_seq, spec3.layers, spec3.hq, spec3.hkv, spec3.d, spec3.block,
                            spec3.W, spec3.B, spec3.K, spec3.R, spec3.lam, wl1.bt_stride, wl1.num_blocks)
    s3, c3 = oracle.scores(sh3, q3, wl1.k, wl1.block_table, wl1.lengths, with_colsum=True)
    np.testing.assert_allclose(c3, G * c1, rtol=1e-13)


def test_group_uses_its_own_heads():
    """Query heads g*G..g*G+G-1 score KV head g: changing head 0's queries leaves group 1 alone."""
    spec = random_spec(34, G=2, hkv=2, W=64, B=16, D=64, n_seq=1, layers=1)
    wl = synth.generate(spec)
    sh = oracle.shape_of(wl)
    s0 = oracle.scores(sh, wl.q, wl.k, wl.block_table, wl.lengths)
    wl.q[:, :, 0] = torch.randn_like(wl.q[:, :, 0].float()).to(torch.bfloat16)
    s1 = oracle.scores(sh, wl.q, wl.k, wl.block_table, wl.lengths)
    assert not np.array_equal(s0[:, :, 0], s1[:, :, 0])
    np.testing.assert_array_equal(s0[:, :, 1], s1[:, :, 1])


def test_buffer_queries_take_part():
    """All W window queries score (the buffer tokens' queries too): change only the last query."""
    spec = random_spec(35, G=1, hkv=1, W=64, B=16, D=64, n_seq=1, layers=1)
    wl = synth.generate(spec)
    sh = oracle.shape_of(wl)
    s0 = oracle.scores(sh, wl.q, wl.k, wl.block_table, wl.lengths)
    wl.q[0, 0, 0, spec.W - 1] = (3 * torch.randn(spec.d)).to(torch.bfloat16)
    s1 = oracle.scores(sh, wl.q, wl.k, wl.block_table, wl.lengths)
    assert np.abs(s0 - s1).max() > 1e-4


def test_no_causal_mask():
    """Key j is scored by queries before it: with queries only at i < j nonzero the score moves."""
    spec = random_spec(36, G=1, hkv=1, W=64, B=16, D=64, n_seq=1, layers=1)
    wl = synth.generate(spec)
    wl.q[0, 0, 0, 1:] = 0                                # only query 0 left
    sh = oracle.shape_of(wl)
    s, cs = oracle.scores(sh, wl.q, wl.k, wl.block_table, wl.lengths, with_colsum=True)
    # query 0 spreads weight over every key j >= 1; zero queries add exactly 1/W each
    extra = cs[0, 0, 0] - (spec.W - 1) / spec.W
    assert np.all(extra[1:] > 0) and abs(extra.sum() - 1.0) < 1e-12


def test_key_permutation_permutes_scores():
    """Swapping two compressible key rows swaps their scores and leaves the rest."""
    spec = random_spec(37, G=2, hkv=1, W=64, B=16, D=64, n_seq=1, layers=1, shuffled=False,
                       len_lo=64, len_hi=64)
    wl = synth.generate(spec)
    sh = oracle.shape_of(wl)
    s0 = oracle.scores(sh, wl.q, wl.k, wl.block_table, wl.lengths)[0, 0, 0]
    a, b = 5, 40                                        # window positions; ws = 0 here
    ka = wl.k[0, a // 16, 0, a % 16].clone()
    wl.k[0, a // 16, 0, a % 16] = wl.k[0, b // 16, 0, b % 16]
    wl.k[0, b // 16, 0, b % 16] = ka
    s1 = oracle.scores(sh, wl.q, wl.k, wl.block_table, wl.lengths)[0, 0, 0]
    perm = np.arange(spec.C)
    perm[a], perm[b] = b, a
    np.testing.assert_allclose(s1, s0[perm], rtol=1e-6)


def test_dominant_key_counts_rows():
    """When every query singles out one key, that key's score is G*W and the rest ~0."""
    spec = random_spec(38, G=2, hkv=1, W=64, B=16, D=64, n_seq=1, layers=1)
    wl = synth.generate(spec)
    L = int(wl.lengths[0])
    jstar = 17
    x = L - spec.W + jstar
    blk = int(wl.block_table[0, x // spec.block])
    wl.k[0, :, 0] = (0.01 * torch.randn_like(wl.k[0, :, 0].float())).to(torch.bfloat16)
    wl.k[0, blk, 0, x % spec.block] = 0
    wl.k[0, blk, 0, x % spec.block, 0] = 32.0
    wl.q.zero_()
    wl.q[..., 0] = 32.0
    s = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths)[0, 0, 0]
    assert s[jstar] == np.float32(2 * spec.W)
    assert np.all(np.delete(s, jstar) < 1e-30)


def test_rejects_short_sequences():
    spec = random_spec(39, W=64)
    wl = synth.generate(spec)
    wl.lengths[0] = 63
    with pytest.raises(ValueError):
        oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths)


def test_tiny_workload_recovers_planted_keys():
    """Soft sanity on the tiny workload: planted keys rank near the top (reported, mild assert)."""
    wl = synth.generate(synth.SPECS["tiny"])
    s = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths)
    assert s.shape == (1, 1, 2, 48)
    np.testing.assert_allclose(s.astype(np.float64).sum(-1) <= 4 * 64, True)
