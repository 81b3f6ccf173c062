"""Pins for the oracle's Top-K and Token2Chunk selection (CPU only)."""
import itertools

import numpy as np
import pytest

import oracle
from _cases import load_golden


def order_key(s, j):
    return (-float(s[j]), j)


def brute_topk(s, K):
    """The unique K-subset whose every member comes before every non-member."""
    C = len(s)
    found = []
    for sub in itertools.combinations(range(C), K):
        ss = set(sub)
        if all(order_key(s, a) < order_key(s, b) for a in ss for b in range(C) if b not in ss):
            found.append(sub)
    assert len(found) == 1
    return list(found[0])


def chunk_den(lam, ln):
    # fmaf(lam, len, 1) rounds once; lam*len + 1 is exact in double for these sizes
    return np.float32(np.float64(np.float32(lam)) * ln + 1.0)


def chunk_scores_independent(s, cand, lam):
    """All index pairs (i < j) of candidates with no candidate strictly between them."""
    cs = set(int(c) for c in cand)
    pairs = []
    for a, b in itertools.combinations(sorted(cs), 2):
        if not any(a < c < b for c in cs):
            pairs.append((a, b))
    out = []
    for a, b in pairs:
        num = np.float32(np.float32(s[a]) + np.float32(s[b]))
        out.append((a, b, np.float32(num / chunk_den(lam, b - a + 1))))
    return out


def greedy_rescan(s, cand, R, lam):
    """A second formulation of the greedy: repeatedly pick the best undecided chunk
    (score desc, left end asc); keep it if its new tokens fit, else reject it.
    Then fill with candidates, then with other positions, both in score order."""
    chunks = chunk_scores_independent(s, cand, lam)
    undecided = list(range(len(chunks)))
    kept = set()
    while undecided:
        best = min(undecided, key=lambda t: (-float(chunks[t][2]), chunks[t][0]))
        undecided.remove(best)
        a, b, _ = chunks[best]
        new = set(range(a, b + 1)) - kept
        if len(kept) + len(new) <= R:
            kept |= new
    order = sorted(range(len(s)), key=lambda j: order_key(s, j))
    cset = set(int(c) for c in cand)
    for j in order:
        if len(kept) >= R:
            break
        if j in cset and j not in kept:
            kept.add(j)
    for j in order:
        if len(kept) >= R:
            break
        if j not in cset and j not in kept:
            kept.add(j)
    return sorted(kept)


def test_hand_worked_token2chunk():
    g = load_golden("token2chunk_hand.json")
    cand, kept, cs, taken = oracle.select(np.asarray(g["scores"], np.float32), g["K"], g["R"], g["lam"],
                                          with_chunks=True)
    assert cand.tolist() == g["expected_cand"]
    np.testing.assert_allclose(cs, g["expected_chunk_scores"], rtol=1e-6)
    assert taken.tolist() == g["expected_chunk_taken"]
    assert kept.tolist() == g["expected_kept"]


@pytest.mark.parametrize("seed", range(40))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    C = int(rng.integers(1, 11))
    s = rng.choice(np.float32([0.5, 1.0, 1.5, 2.0, 0.25]), size=C)    # forces ties
    for K in range(1, C + 1):
        cand, _ = oracle.select(s, K, 1, 0.1)
        assert cand.tolist() == sorted(brute_topk(s, K))


@pytest.mark.parametrize("seed", range(30))
def test_chunks_enumerated(seed):
    rng = np.random.default_rng(100 + seed)
    C = int(rng.integers(4, 40))
    K = int(rng.integers(2, C + 1))
    s = rng.random(C).astype(np.float32)
    lam = float(rng.choice([0.1, 0.5, 0.0, 2.0]))
    cand, _, cs, _ = oracle.select(s, K, 1, lam, with_chunks=True)
    ind = chunk_scores_independent(s, cand, lam)
    assert len(ind) == K - 1
    assert [(a, b) for a, b, _ in ind] == [(int(cand[t]), int(cand[t + 1])) for t in range(K - 1)]
    np.testing.assert_array_equal(cs, np.asarray([c for _, _, c in ind], np.float32))


def test_chunk_score_uses_only_endpoints_and_length():
    rng = np.random.default_rng(7)
    s = rng.random(30).astype(np.float32) + 1.0
    cand, _, cs0, _ = oracle.select(s, 6, 10, 0.1, with_chunks=True)
    s2 = s.copy()
    inner = [j for j in range(30) if j not in set(cand.tolist())]
    s2[inner] = rng.random(len(inner)).astype(np.float32) * 0.5       # still below every candidate
    cand2, _, cs2, _ = oracle.select(s2, 6, 10, 0.1, with_chunks=True)
    assert cand.tolist() == cand2.tolist()
    np.testing.assert_array_equal(cs0, cs2)


@pytest.mark.parametrize("seed", range(60))
def test_greedy_matches_rescan_formulation(seed):
    rng = np.random.default_rng(200 + seed)
    C = int(rng.integers(2, 120))
    K = int(rng.integers(1, min(C, 40) + 1))
    R = int(rng.integers(1, C + 1))
    if seed % 3 == 0:
        s = rng.choice(np.float32([1.0, 2.0, 3.0, 4.0]), size=C)       # chunk-score ties too
    else:
        s = rng.exponential(size=C).astype(np.float32)
    lam = float(rng.choice([0.1, 0.3]))
    _, kept = oracle.select(s, K, R, lam)
    assert kept.tolist() == greedy_rescan(s, oracle.select(s, K, R, lam)[0], R, lam)


@pytest.mark.parametrize("seed", range(10))
def test_k1_is_textbook_top_r(seed):
    rng = np.random.default_rng(300 + seed)
    C, R = 50, int(rng.integers(1, 50))
    s = rng.choice(np.float32([1, 2, 3, 5, 8]), size=C)
    _, kept = oracle.select(s, 1, R, 0.1)
    top = sorted(range(C), key=lambda j: order_key(s, j))[:R]
    assert kept.tolist() == sorted(top)


def test_budget_covering_the_span_keeps_it_whole():
    rng = np.random.default_rng(9)
    C, K = 80, 5
    s = rng.random(C).astype(np.float32)
    cand, _ = oracle.select(s, K, 1, 0.1)
    span = int(cand[-1] - cand[0] + 1)
    R = span + 7
    _, kept = oracle.select(s, K, R, 0.1)
    inside = set(range(int(cand[0]), int(cand[-1]) + 1))
    assert inside <= set(kept.tolist())
    rest = [j for j in sorted(range(C), key=lambda j: order_key(s, j)) if j not in inside][:7]
    assert set(kept.tolist()) == inside | set(rest)


def test_adjacent_candidates_make_length_two_chunks():
    s = np.float32([0.0, 5.0, 4.0, 0.0, 0.0, 3.0])
    cand, kept, cs, taken = oracle.select(s, 3, 2, 0.5, with_chunks=True)
    assert cand.tolist() == [1, 2, 5]
    assert cs[0] == np.float32(9.0) / chunk_den(0.5, 2)
    assert taken.tolist() == [True, False] and kept.tolist() == [1, 2]


@pytest.mark.parametrize("seed", range(20))
def test_invariants(seed):
    rng = np.random.default_rng(400 + seed)
    C = int(rng.integers(1, 300))
    K = int(rng.integers(1, C + 1))
    R = int(rng.integers(1, C + 1))
    s = rng.random(C).astype(np.float32)
    cand, kept = oracle.select(s, K, R, 0.1)
    assert len(kept) == R and np.all(np.diff(kept) > 0) and kept[0] >= 0 and kept[-1] < C
    assert len(cand) == K and np.all(np.diff(cand) > 0)


def test_greedy_vs_exhaustive_knapsack_is_information_only():
    """On tiny windows report how close first fit comes to the best chunk subset."""
    rng = np.random.default_rng(11)
    ratios = []
    for _ in range(20):
        C, K, R = 16, 6, 8
        s = rng.random(C).astype(np.float32)
        cand, _, cs, taken = oracle.select(s, K, R, 0.1, with_chunks=True)
        best = 0.0
        for mask in range(1 << (K - 1)):
            toks = set()
            val = 0.0
            for t in range(K - 1):
                if mask >> t & 1:
                    toks |= set(range(int(cand[t]), int(cand[t + 1]) + 1))
                    val += float(cs[t])
            if len(toks) <= R:
                best = max(best, val)
        got = float(np.sum(cs[taken]))
        ratios.append(got / best if best > 0 else 1.0)
    assert min(ratios) > 0.0 and max(ratios) <= 1.0 + 1e-6


def test_rejects_bad_budgets():
    s = np.ones(10, np.float32)
    for K, R in [(0, 1), (11, 1), (1, 0), (1, 11)]:
        with pytest.raises(ValueError):
            oracle.select(s, K, R, 0.1)


def test_batch_equals_single():
    rng = np.random.default_rng(5)
    sc = rng.random((3, 4, 100)).astype(np.float32)
    cand, kept = oracle.select_batch(sc, 10, 30, 0.1)
    for i in range(3):
        for j in range(4):
            c1, k1 = oracle.select(sc[i, j], 10, 30, 0.1)
            assert cand[i, j].tolist() == c1.tolist() and kept[i, j].tolist() == k1.tolist()
