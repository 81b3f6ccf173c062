"""Pins for the oracle's ablation variants (CPU only): causal window scores and
the two selection modes that replace Token2Chunk (token-level Top-R and
fixed-size chunks).

Each check ties the variant to something outside the oracle: a library softmax
with a causal mask, a harmonic-number closed form, a brute-force sort, or an
identity with the main selection path that holds by definition.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import independent_colsum, random_spec


# ---- causal scores -----------------------------------------------------------

@pytest.mark.parametrize("seed,G,W,B,D,block", [
    (41, 1, 64, 16, 64, 16), (42, 2, 48, 8, 32, 16), (43, 3, 32, 4, 16, 8), (44, 2, 128, 16, 128, 16)])
def test_causal_matches_masked_fp64_softmax(seed, G, W, B, D, block):
    """Library softmax (torch fp64) with keys after the query masked out."""
    spec = random_spec(seed, G=G, W=W, B=B, D=D, block=block)
    wl = synth.generate(spec)
    s, cs = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths, with_colsum=True,
                          causal=True)
    ref = independent_colsum(wl, causal=True)
    np.testing.assert_allclose(cs, ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(s, ref[..., :spec.C].astype(np.float32), rtol=2 ** -23, atol=0)
    # the mask matters: the bidirectional scores differ
    assert not np.allclose(cs, independent_colsum(wl), rtol=1e-6)


def test_causal_zero_queries_harmonic_closed_form():
    """Q = 0: query i spreads weight 1/(i+1) over keys 0..i, so
    t[j] = G * sum_{i=j}^{W-1} 1/(i+1) = G * (H_W - H_j)."""
    spec = random_spec(45, G=3, W=64, B=16, D=32)
    wl = synth.generate(spec)
    wl.q.zero_()
    s, cs = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths, with_colsum=True,
                          causal=True)
    W = spec.W
    H = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, W + 1))])   # H[n] = sum_{k<=n} 1/k
    want = 3 * (H[W] - H[np.arange(W)])
    np.testing.assert_allclose(cs.reshape(-1, W), np.broadcast_to(want, (cs.size // W, W)), rtol=1e-13)
    assert cs[..., -1].ravel()[0] == pytest.approx(3.0 / W, rel=1e-13)


@pytest.mark.parametrize("seed", [46, 47])
def test_causal_row_sums(seed):
    spec = random_spec(seed, G=2, W=64, B=24, D=32, plant="bernoulli")
    wl = synth.generate(spec)
    s, cs = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths, with_colsum=True,
                          causal=True)
    np.testing.assert_allclose(cs.sum(-1), 2 * spec.W, rtol=1e-12)
    # key 0 collects the whole first row of every head
    assert np.all(cs[..., 0] >= 2 - 1e-12)


# ---- selection modes -----------------------------------------------------------

def brute_top(s, R):
    """The R positions first under (score desc, index asc), by a full sort."""
    order = sorted(range(len(s)), key=lambda j: (-float(s[j]), j))
    return np.sort(np.asarray(order[:R], np.int32))


@pytest.mark.parametrize("seed,C,K,R", [(51, 40, 8, 12), (52, 100, 16, 30), (53, 7, 3, 7), (54, 64, 64, 5)])
def test_top_r_is_brute_force_top(seed, C, K, R):
    rng = np.random.default_rng(seed)
    s = rng.integers(0, 6, C).astype(np.float32) / 4          # many ties
    cand, kept = oracle.select_mode(s, K, R, 0.1, oracle.SELECT_TOP_R)
    np.testing.assert_array_equal(kept, brute_top(s, R))
    cand0, _ = oracle.select(s, K, R, 0.1)
    np.testing.assert_array_equal(cand, cand0)                 # candidates unchanged


@pytest.mark.parametrize("seed", [55, 56, 57])
def test_top_r_is_token2chunk_with_one_candidate(seed):
    """With K = 1 Token2Chunk has no chunk, so its fills reduce to the top R."""
    s = np.random.default_rng(seed).standard_normal(50).astype(np.float32)
    _, k1 = oracle.select(s, 1, 17, 0.1)
    _, kr = oracle.select_mode(s, 1, 17, 0.1, oracle.SELECT_TOP_R)
    np.testing.assert_array_equal(k1, kr)


@pytest.mark.parametrize("chunk", [1, 50])
def test_fixed_chunks_degenerate_to_top_r(chunk):
    """chunk = 1: every chunk is one token and its mean is its score; chunk = C:
    the single chunk does not fit R < C, so the fill takes the top R."""
    s = np.random.default_rng(58).integers(0, 9, 50).astype(np.float32)
    _, kf = oracle.select_mode(s, 4, 13, 0.1, oracle.SELECT_FIXED_CHUNK, chunk)
    np.testing.assert_array_equal(kf, brute_top(s, 13))


def test_fixed_chunks_hand_worked():
    """C = 10, chunk 4: chunks [0,4) [4,8) [8,10) with means 1.0, 2.5, 3.0.
    Visit order 2, 1, 0.  R = 6: chunk 2 (2 tokens) fits, chunk 1 (4 more -> 6)
    fits, chunk 0 does not: kept = 4..9."""
    s = np.asarray([1, 1, 1, 1, 2, 3, 2, 3, 3, 3], np.float32)
    _, kept = oracle.select_mode(s, 2, 6, 0.1, oracle.SELECT_FIXED_CHUNK, 4)
    np.testing.assert_array_equal(kept, [4, 5, 6, 7, 8, 9])
    # R = 5: chunk 2 fits (2), chunk 1 does not (6 > 5), chunk 0 does not (6 > 5);
    # the fill then takes the 3 best other positions: 5, 7 (score 3), then 4 (score 2, lower index)
    _, kept = oracle.select_mode(s, 2, 5, 0.1, oracle.SELECT_FIXED_CHUNK, 4)
    np.testing.assert_array_equal(kept, [4, 5, 7, 8, 9])


@pytest.mark.parametrize("seed", [61, 62])
def test_fixed_chunks_take_the_best_whole_chunks(seed):
    """C and R multiples of the chunk, well separated means: kept is exactly the
    union of the R/chunk chunks with the largest means (computed in fp64)."""
    rng = np.random.default_rng(seed)
    chunk, nch, take = 8, 12, 4
    level = rng.permutation(nch).astype(np.float64)           # distinct chunk levels
    s = (np.repeat(level, chunk) + rng.uniform(0, 0.1, nch * chunk)).astype(np.float32)
    _, kept = oracle.select_mode(s, 5, take * chunk, 0.1, oracle.SELECT_FIXED_CHUNK, chunk)
    means = s.astype(np.float64).reshape(nch, chunk).mean(1)
    best = np.sort(np.argsort(-means)[:take])
    want = (best[:, None] * chunk + np.arange(chunk)[None, :]).ravel()
    np.testing.assert_array_equal(kept, want)


@pytest.mark.parametrize("mode,chunk", [(1, 0), (2, 3), (2, 16)])
def test_mode_invariants(mode, chunk):
    rng = np.random.default_rng(63 + chunk)
    for C, K, R in [(30, 5, 7), (200, 20, 60), (33, 33, 33)]:
        s = rng.standard_normal(C).astype(np.float32)
        cand, kept = oracle.select_mode(s, K, R, 0.1, mode, min(chunk, C) or 0)
        assert len(kept) == R and np.all(np.diff(kept) > 0) and kept[0] >= 0 and kept[-1] < C
        assert len(cand) == K and np.all(np.diff(cand) > 0)


def test_mode_batch_matches_single():
    rng = np.random.default_rng(64)
    sc = rng.standard_normal((3, 4, 40)).astype(np.float32)
    for mode, chunk in [(0, 0), (1, 0), (2, 5)]:
        cb, kb = oracle.select_mode_batch(sc, 6, 11, 0.1, mode, chunk)
        for idx in np.ndindex(3, 4):
            c1, k1 = oracle.select_mode(sc[idx], 6, 11, 0.1, mode, chunk)
            np.testing.assert_array_equal(cb[idx], c1)
            np.testing.assert_array_equal(kb[idx], k1)


def test_mode_rejects_bad_arguments():
    s = np.zeros(10, np.float32)
    for mode, chunk in [(3, 0), (2, 0), (2, 11), (-1, 0)]:
        with pytest.raises(ValueError):
            oracle.select_mode(s, 2, 3, 0.1, mode, chunk)
