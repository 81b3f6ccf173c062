"""GPU parity of the window-query ring: kara_compact_queries bit-exact against
the oracle, its transactional and error paths, kara_append_queries, and two
compressions in a row that score from the ring."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import random_spec
from _gpu import SCORE_RTOL, lib, rel_err, to_device
from test_oracle_qring import make_ring, random_kept

pytestmark = pytest.mark.gpu


def ring_call(kara, wl, ring_np, kept_np, err_value=0):
    sp = wl.spec
    d = to_device(wl)
    ring = torch.from_numpy(ring_np.view(np.int16)).cuda().view(torch.bfloat16)
    c = kara.cache(d.k, d.v, sp.hq)
    p = kara.params(sp.W, sp.B, sp.K, sp.R, sp.lam)
    b = kara.batch(d.lengths, d.block_table, ring)
    err = torch.full((1,), err_value, dtype=torch.int32, device="cuda")
    kara.kara_compact_queries(c, p, b, torch.from_numpy(kept_np).cuda(), err)
    torch.cuda.synchronize()
    return ring.view(torch.int16).cpu().numpy().view(np.uint16), int(err.item())


@pytest.mark.parametrize("seed,G,W,B,R,D", [
    (91, 2, 64, 16, 20, 64), (92, 4, 256, 32, 120, 128), (93, 1, 2048, 256, 500, 128), (94, 3, 128, 0, 7, 64)])
def test_compact_queries_matches_oracle(seed, G, W, B, R, D):
    kara = lib()
    sp = random_spec(seed, G=G, W=W, B=B, D=D, n_seq=3, layers=2, len_lo=W, len_hi=W + 300, R=R)
    wl = synth.generate(sp)
    rng = np.random.default_rng(seed)
    _, ring = make_ring(wl, rng)
    kept = random_kept(sp, rng)
    got, err = ring_call(kara, wl, ring, kept)
    assert err == 0
    want = oracle.compact_queries(oracle.shape_of(wl), ring, wl.lengths, kept)
    assert np.array_equal(got, want)


def test_failed_step_moves_nothing_and_bad_kept_is_reported():
    kara = lib()
    sp = random_spec(95, G=2, W=64, B=16, D=64, n_seq=2, layers=1, R=20)
    wl = synth.generate(sp)
    rng = np.random.default_rng(95)
    _, ring = make_ring(wl, rng)
    kept = random_kept(sp, rng)
    got, err = ring_call(kara, wl, ring, kept, err_value=kara.ENOBLOCKS)
    assert err == kara.ENOBLOCKS and np.array_equal(got, ring)
    bad = kept.copy()
    bad[1, 0, 1, 3] = bad[1, 0, 1, 2]             # not strictly increasing
    got, err = ring_call(kara, wl, ring, bad)
    assert err == kara.EINVAL
    want = oracle.compact_queries(oracle.shape_of(wl), ring, wl.lengths, kept)
    assert np.array_equal(got[1, 0, 2:4], ring[1, 0, 2:4])      # the heads of that window are untouched
    assert np.array_equal(got[0], want[0])                     # other windows are compacted


def test_append_writes_row_len_mod_w():
    kara = lib()
    sp = random_spec(96, G=2, W=64, B=16, D=128, n_seq=3, layers=2, len_lo=64, len_hi=200)
    wl = synth.generate(sp)
    d = to_device(wl)
    ring = torch.zeros(sp.n_seq, sp.layers, sp.hq, sp.W, sp.d, dtype=torch.bfloat16, device="cuda")
    q_new = torch.randn(sp.n_seq, sp.layers, sp.hq, sp.d, device="cuda").to(torch.bfloat16)
    c = kara.cache(d.k, d.v, sp.hq)
    kara.kara_append_queries(c, kara.params(sp.W, sp.B, sp.K, sp.R, sp.lam), kara.batch(d.lengths, d.block_table, ring),
                             q_new)
    want = torch.zeros_like(ring)
    for s in range(sp.n_seq):
        want[s, :, :, int(wl.lengths[s]) % sp.W] = q_new[s]
    assert torch.equal(ring, want)


def test_two_compressions_score_from_the_ring():
    """Compress, move the queries, decode C - R + 9 tokens into the ring and the
    cache, compress again: both events score from the ring and match the oracle
    on the position-ordered window."""
    kara = lib()
    from decode_kv_cache_03_gb300 import Compressor
    from decode_kv_cache_03_gb300.periodic import BlockPool, append_tokens
    sp = random_spec(97, G=2, W=128, B=16, D=128, n_seq=3, layers=2, len_lo=300, len_hi=420, K=8, R=30,
                     plant="bernoulli")
    wl = synth.generate(sp, extra_fresh_per_seq=40)
    d = to_device(wl)
    rng = np.random.default_rng(97)
    _, ring_np = make_ring(wl, rng)
    ring = torch.from_numpy(ring_np.view(np.int16)).cuda().view(torch.bfloat16)
    comp = Compressor(d.k, d.v, sp.hq, sp.W, sp.B, sp.K, sp.R, sp.lam)
    stride = wl.bt_stride + 8
    table = torch.full((sp.n_seq, stride), -1, dtype=torch.int32)
    table[:, :wl.bt_stride] = wl.block_table
    lengths = wl.lengths.tolist()
    pool = BlockPool(wl.fresh.tolist())
    gen = torch.Generator(device="cuda").manual_seed(4)
    for event in range(2):
        # the window queries in position order, read back from the ring, for the oracle
        L = torch.tensor(lengths, dtype=torch.int32)
        q_log = torch.empty(sp.n_seq, sp.layers, sp.hq, sp.W, sp.d, dtype=torch.bfloat16)
        rc = ring.cpu()
        for s in range(sp.n_seq):
            rows = (int(L[s]) - sp.W + torch.arange(sp.W)) % sp.W
            q_log[s] = rc[s][:, :, rows]
        kh = d.k.view(torch.int16).cpu().numpy().view(np.uint16)
        sh = oracle.make_shape(sp.n_seq, sp.layers, sp.hq, sp.hkv, sp.d, sp.block, sp.W, sp.B, sp.K, sp.R, sp.lam,
                               stride, wl.num_blocks)
        ref = oracle.scores(sh, q_log, kh, table.numpy(), L.numpy())
        # the step, reading the ring
        nn, no, tn, to = comp.plan(L, stride)
        fresh = torch.tensor(pool.take(tn), dtype=torch.int32, device="cuda")
        d_bt = table.cuda()
        d_len = L.cuda()
        freed = torch.empty(max(to, 1), dtype=torch.int32, device="cuda")
        new_len = torch.empty(sp.n_seq, dtype=torch.int32, device="cuda")
        scores = torch.empty(sp.n_seq, sp.layers, sp.hkv, sp.C, device="cuda")
        kept = torch.empty(sp.n_seq, sp.layers, sp.hkv, sp.R, dtype=torch.int32, device="cuda")
        comp.compress(d_len, d_bt, ring, fresh, freed, new_len, scores=scores, kept=kept)
        b = kara.batch(d_len, d_bt, ring)
        kara.kara_compact_queries(comp.cache, comp.params, b, kept, comp.err)
        assert comp.error() == 0
        assert rel_err(scores.cpu().numpy(), ref).max() <= SCORE_RTOL
        _, k_o = oracle.select_batch(scores.cpu().numpy(), sp.K, sp.R, sp.lam)
        assert np.array_equal(kept.cpu().numpy(), k_o)
        want_ring = oracle.compact_queries(sh, ring_np_from(rc), L, k_o)
        assert np.array_equal(ring.view(torch.int16).cpu().numpy().view(np.uint16), want_ring)
        table[:] = d_bt.cpu()
        lengths = new_len.cpu().tolist()
        pool.give(freed[:to].cpu().tolist())
        # decode: every sequence appends C - R + 9 tokens (K, V and the query)
        for _ in range(sp.C - sp.R + 9):
            before = list(lengths)
            append_tokens(lengths, table, pool, sp.block)
            for s in range(sp.n_seq):
                x = before[s]
                blk, slot = int(table[s, x // sp.block]), x % sp.block
                d.k[:, blk, :, slot] = torch.randn(sp.layers, sp.hkv, sp.d, generator=gen, device="cuda").to(torch.bfloat16)
                d.v[:, blk, :, slot] = torch.randn(sp.layers, sp.hkv, sp.d, generator=gen, device="cuda").to(torch.bfloat16)
            q_new = torch.randn(sp.n_seq, sp.layers, sp.hq, sp.d, generator=gen, device="cuda").to(torch.bfloat16)
            kara.kara_append_queries(comp.cache, comp.params,
                                     kara.batch(torch.tensor(before, dtype=torch.int32).cuda(), d_bt, ring), q_new)


def ring_np_from(ring_cpu):
    return ring_cpu.view(torch.int16).numpy().view(np.uint16)
