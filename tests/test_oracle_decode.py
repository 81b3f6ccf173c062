"""Pins for the oracle's decode attention over the paged cache (CPU only):
a library fp64 softmax over a numpy gather, closed forms (zero query, one
cached token, a dominant key), and the compacted cache read back through the
rewritten table against a direct gather of the rows the step keeps."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import random_spec


def gathered(wl, pool, s, layer, g, positions):
    """Rows of logical positions of sequence s, gathered through the block table with numpy."""
    sp = wl.spec
    bt = wl.block_table.numpy()
    blk = bt[s, positions // sp.block]
    return pool.float().double().numpy()[layer, blk, g, positions % sp.block, :]


def independent_decode(wl, q, layer, lengths=None, block_table=None, k=None, v=None):
    sp = wl.spec
    G = sp.hq // sp.hkv
    lengths = wl.lengths if lengths is None else lengths
    wl2 = synth.Workload(sp, wl.q, wl.k if k is None else k, wl.v if v is None else v, lengths,
                         wl.block_table if block_table is None else block_table, wl.fresh, wl.prefix_pool,
                         wl.fresh_base)
    out = np.zeros((sp.n_seq, sp.hq, sp.d))
    for s in range(sp.n_seq):
        pos = np.arange(int(lengths[s]))
        for h in range(sp.hq):
            kk = torch.from_numpy(gathered(wl2, wl2.k, s, layer, h // G, pos))
            vv = torch.from_numpy(gathered(wl2, wl2.v, s, layer, h // G, pos))
            p = torch.softmax(kk @ q[s, h].double() / np.sqrt(sp.d), dim=0)
            out[s, h] = (p @ vv).numpy()
    return out


@pytest.mark.parametrize("seed,G,D,layer", [(71, 1, 64, 0), (72, 4, 128, 1), (73, 3, 32, 1), (74, 8, 128, 0)])
def test_decode_matches_library_softmax(seed, G, D, layer):
    spec = random_spec(seed, G=G, W=64, B=16, D=D, len_lo=20, len_hi=300)
    wl = synth.generate(spec)
    q = synth.decode_queries(spec, seed)
    out = oracle.decode_attention(oracle.shape_of(wl), layer, q, wl.k, wl.v, wl.block_table, wl.lengths)
    ref = independent_decode(wl, q, layer)
    np.testing.assert_allclose(out, ref.astype(np.float32), rtol=1e-6, atol=1e-7)


def test_zero_query_is_the_mean_of_v():
    spec = random_spec(75, G=2, W=64, B=16, D=64, len_lo=40, len_hi=200)
    wl = synth.generate(spec)
    q = torch.zeros(spec.n_seq, spec.hq, spec.d, dtype=torch.bfloat16)
    out = oracle.decode_attention(oracle.shape_of(wl), 1, q, wl.k, wl.v, wl.block_table, wl.lengths)
    for s in range(spec.n_seq):
        pos = np.arange(int(wl.lengths[s]))
        for h in range(spec.hq):
            want = gathered(wl, wl.v, s, 1, h // 2, pos).mean(0)
            np.testing.assert_allclose(out[s, h], want, rtol=1e-6, atol=1e-7)


def test_one_cached_token_returns_its_value_row():
    spec = random_spec(76, G=2, W=64, B=16, D=64)
    wl = synth.generate(spec)
    lengths = torch.ones_like(wl.lengths)
    q = synth.decode_queries(spec, 1)
    out = oracle.decode_attention(oracle.shape_of(wl), 0, q, wl.k, wl.v, wl.block_table, lengths)
    for s in range(spec.n_seq):
        for h in range(spec.hq):
            np.testing.assert_array_equal(out[s, h], gathered(wl, wl.v, s, 0, h // 2, np.array([0]))[0])


def test_dominant_key_takes_all_the_weight():
    spec = random_spec(77, G=1, hkv=2, W=64, B=16, D=64, len_lo=100, len_hi=100)
    wl = synth.generate(spec)
    x = 37
    q = torch.zeros(spec.n_seq, spec.hq, spec.d, dtype=torch.bfloat16)
    for s in range(spec.n_seq):
        for h in range(spec.hq):
            q[s, h] = torch.from_numpy(gathered(wl, wl.k, s, 0, h, np.array([x]))[0] * 8)
    out = oracle.decode_attention(oracle.shape_of(wl), 0, q, wl.k, wl.v, wl.block_table, wl.lengths)
    for s in range(spec.n_seq):
        for h in range(spec.hq):
            np.testing.assert_allclose(out[s, h], gathered(wl, wl.v, s, 0, h, np.array([x]))[0], atol=1e-6)


def test_reads_the_compacted_cache_through_the_rewritten_table():
    """After compaction, decode attention over the new table equals decode
    attention over the logical rows the step keeps, gathered from the old cache:
    the head of the partial block, the kept rows, then the protected buffer."""
    spec = random_spec(78, G=2, W=64, B=16, D=64, len_lo=80, len_hi=250, K=6, R=20)
    wl = synth.generate(spec)
    sc = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths)
    _, kept = oracle.select_batch(sc, spec.K, spec.R, spec.lam)
    kh = wl.k.view(torch.int16).numpy().view(np.uint16)
    vh = wl.v.view(torch.int16).numpy().view(np.uint16)
    st, k2, v2, bt2, _, nl2 = oracle.compact(oracle.shape_of(wl), kh, vh, wl.block_table, wl.lengths, kept,
                                             wl.fresh)
    assert st == oracle.OK
    q = synth.decode_queries(spec, 2)
    layer = 1
    out = oracle.decode_attention(oracle.shape_of(wl), layer, q, torch.from_numpy(k2.view(np.int16)),
                                  torch.from_numpy(v2.view(np.int16)), bt2, nl2)
    G = spec.hq // spec.hkv
    for s in range(spec.n_seq):
        L = int(wl.lengths[s])
        ws = L - spec.W
        for h in range(spec.hq):
            g = h // G
            pos = np.concatenate([np.arange(ws), ws + kept[s, layer, g], np.arange(L - spec.B, L)])
            kk = torch.from_numpy(gathered(wl, wl.k, s, layer, g, pos))
            vv = torch.from_numpy(gathered(wl, wl.v, s, layer, g, pos))
            p = torch.softmax(kk @ q[s, h].double() / np.sqrt(spec.d), dim=0)
            np.testing.assert_allclose(out[s, h], (p @ vv).numpy(), rtol=1e-6, atol=1e-7)


def test_rejects_short_or_overlong_lengths():
    spec = random_spec(79, G=2, W=64, B=16, D=64)
    wl = synth.generate(spec)
    q = synth.decode_queries(spec)
    for bad in (0, wl.bt_stride * spec.block + 1):
        ln = wl.lengths.clone()
        ln[0] = bad
        with pytest.raises(ValueError):
            oracle.decode_attention(oracle.shape_of(wl), 0, q, wl.k, wl.v, wl.block_table, ln)
