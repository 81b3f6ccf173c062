"""GPU parity of decode attention over the paged cache against the oracle,
including the cache a compression call has just rewritten.

Tolerance: the logits are fp32 sums of exact bf16 products (relative error
about D * 2^-24); each weight enters the weighted sum as two bf16 terms
(relative error about 2^-17) and the sums are fp32 over at most a few thousand
rows, so for unit-scale V the output is within 1e-4 absolute of the fp64
result; the test allows 2e-4 absolute plus 1e-3 relative."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import random_spec
from _gpu import lib, run_compress, to_device

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-4, 1e-3


def run_decode(kara, k, v, hq, layer, lengths, bt, q):
    c = kara.cache(k, v, hq)
    n, bt_stride = bt.shape
    ws = torch.empty(kara.kara_decode_workspace_size(c, n, bt_stride), dtype=torch.uint8, device="cuda")
    out = torch.full((n, hq, k.shape[-1]), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kara.kara_decode_attention(c, layer, lengths, bt, q, out, ws, err)
    return out.cpu().numpy(), kara.kara_get_error(err)


@pytest.mark.parametrize("G,D,len_lo,len_hi", [
    (1, 64, 1, 40), (2, 64, 100, 700), (4, 128, 20, 600), (5, 128, 1500, 2100), (8, 128, 500, 1100),
    (3, 64, 1023, 1026), (6, 128, 2047, 2049), (7, 128, 1, 1)])
def test_decode_matches_oracle(G, D, len_lo, len_hi):
    """Lengths below, at and across the 1024-key split, one cached token, and G = 1..8."""
    kara = lib()
    spec = random_spec(500 + G * D + len_lo, G=G, hkv=2, W=64, B=16, D=D, n_seq=4, layers=2,
                       len_lo=max(len_lo, 64), len_hi=max(len_hi, 64))
    wl = synth.generate(spec)
    if len_hi < 64:   # shorter than any window: keep the first len tokens of each table
        gen = torch.Generator().manual_seed(len_hi)
        wl.lengths.copy_(torch.randint(len_lo, len_hi + 1, (spec.n_seq,), generator=gen, dtype=torch.int32))
    q = synth.decode_queries(spec, G)
    d = to_device(wl)
    for layer in (0, 1):
        got, st = run_decode(kara, d.k, d.v, wl.spec.hq, layer, d.lengths, d.block_table, q.cuda())
        assert st == 0
        ref = oracle.decode_attention(oracle.shape_of(wl), layer, q, wl.k, wl.v, wl.block_table, wl.lengths)
        np.testing.assert_allclose(got, ref, atol=ATOL, rtol=RTOL)


def test_decode_reads_the_table_compression_rewrote():
    """Compress, then decode over the rewritten table and shorter lengths: the
    same result as the oracle decoding the oracle's compacted cache."""
    kara = lib()
    spec = random_spec(510, G=4, hkv=2, W=256, B=32, D=128, n_seq=3, layers=2, len_lo=600, len_hi=1500, K=16,
                       R=60, plant="bernoulli")
    wl = synth.generate(spec)
    d = to_device(wl)
    out = run_compress(d)
    assert out["status"] == 0
    kh = wl.k.view(torch.int16).numpy().view(np.uint16)
    vh = wl.v.view(torch.int16).numpy().view(np.uint16)
    st, k2, v2, bt2, _, nl2 = oracle.compact(oracle.shape_of(wl), kh, vh, wl.block_table, wl.lengths, out["kept"],
                                             wl.fresh)
    assert st == oracle.OK and np.array_equal(out["bt"], bt2) and np.array_equal(out["new_len"], nl2)
    q = synth.decode_queries(spec, 9)
    for layer in (0, 1):
        got, st = run_decode(kara, d.k, d.v, spec.hq, layer, torch.from_numpy(nl2).cuda(),
                             torch.from_numpy(bt2).cuda().contiguous(), q.cuda())
        assert st == 0
        ref = oracle.decode_attention(oracle.shape_of(wl), layer, q, torch.from_numpy(k2.view(np.int16)),
                                      torch.from_numpy(v2.view(np.int16)), bt2, nl2)
        np.testing.assert_allclose(got, ref, atol=ATOL, rtol=RTOL)


def test_decode_on_device_right_after_compress():
    """Compress, then decode every layer on the same stream from the device-side
    new lengths and the table the step rewrote in place (no host step between):
    the oracle's decode of the oracle's compacted cache."""
    from decode_kv_cache_03_gb300.compressor import Compressor
    spec = random_spec(511, G=4, hkv=2, W=256, B=32, D=128, n_seq=3, layers=2, len_lo=600, len_hi=1500, K=16,
                       R=60, plant="bernoulli")
    wl = synth.generate(spec)
    d = to_device(wl)
    comp = Compressor(d.k, d.v, spec.hq, spec.W, spec.B, spec.K, spec.R, spec.lam)
    _, _, _, to = comp.plan(wl.lengths, wl.bt_stride)
    bt = d.block_table.clone()
    freed = torch.empty(to, dtype=torch.int32, device="cuda")
    new_len = torch.empty(spec.n_seq, dtype=torch.int32, device="cuda")
    kept = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.R, dtype=torch.int32, device="cuda")
    q = synth.decode_queries(spec, 10).cuda()
    outs = [torch.full((spec.n_seq, spec.hq, spec.d), float("nan"), device="cuda") for _ in range(spec.layers)]
    comp.compress(d.lengths, bt, d.q, d.fresh, freed, new_len, kept=kept)
    for layer in range(spec.layers):
        comp.decode(layer, new_len, bt, q, outs[layer])
    assert comp.error() == 0
    kh = wl.k.view(torch.int16).numpy().view(np.uint16)
    vh = wl.v.view(torch.int16).numpy().view(np.uint16)
    st, k2, v2, bt2, _, nl2 = oracle.compact(oracle.shape_of(wl), kh, vh, wl.block_table, wl.lengths,
                                             kept.cpu().numpy(), wl.fresh)
    assert st == oracle.OK
    for layer in range(spec.layers):
        ref = oracle.decode_attention(oracle.shape_of(wl), layer, q.cpu(), torch.from_numpy(k2.view(np.int16)),
                                      torch.from_numpy(v2.view(np.int16)), bt2, nl2)
        np.testing.assert_allclose(outs[layer].cpu().numpy(), ref, atol=ATOL, rtol=RTOL)


def test_decode_reports_bad_lengths_and_blocks():
    kara = lib()
    spec = random_spec(511, G=2, hkv=2, W=64, B=16, D=64, n_seq=3, layers=1, len_lo=100, len_hi=200)
    wl = synth.generate(spec)
    d = to_device(wl)
    q = synth.decode_queries(spec).cuda()
    ln = d.lengths.clone()
    ln[1] = 0
    got, st = run_decode(kara, d.k, d.v, spec.hq, 0, ln, d.block_table, q)
    assert st == kara.EINVAL and np.all(got[1] == 0) and np.all(np.isfinite(got))
    bt = d.block_table.clone()
    bt[2, 1] = wl.num_blocks + 5      # outside the pool: reported, never dereferenced
    got, st = run_decode(kara, d.k, d.v, spec.hq, 0, d.lengths, bt, q)
    assert st == kara.EBADBLOCK


@pytest.mark.parametrize("D", [64, 128])
def test_decode_ignores_rows_past_the_end(D):
    """The last block of each sequence holds rows past its length; they are
    NaN here and must not reach the output (the oracle reads x < L only)."""
    kara = lib()
    spec = random_spec(520 + D, G=4, hkv=2, W=64, B=16, D=D, n_seq=4, layers=1, len_lo=1031, len_hi=1100)
    wl = synth.generate(spec)
    gen = torch.Generator().manual_seed(D)
    short = torch.randint(65, 1031, (spec.n_seq,), generator=gen, dtype=torch.int32)
    wl.lengths.copy_(torch.minimum(wl.lengths, short))  # shorter than generated: the table covers them
    wl.lengths[0] = 1024 + 7                    # a ragged block right after the split boundary
    k, v = wl.k.clone(), wl.v.clone()
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    for s in range(spec.n_seq):
        L = int(wl.lengths[s])
        if L % 16:
            blk = int(wl.block_table[s, L // 16])
            k[0, blk, :, L % 16:] = nan
            v[0, blk, :, L % 16:] = nan
    q = synth.decode_queries(spec, 3)
    d = to_device(wl)
    got, st = run_decode(kara, k.cuda(), v.cuda(), spec.hq, 0, d.lengths, d.block_table, q.cuda())
    assert st == 0 and np.all(np.isfinite(got))
    ref = oracle.decode_attention(oracle.shape_of(wl), 0, q, k, v, wl.block_table, wl.lengths)
    np.testing.assert_allclose(got, ref, atol=ATOL, rtol=RTOL)


def test_decode_reads_a_bad_block_as_zeros():
    """A block id outside the pool is reported and its rows read as zeros: the
    same result as the oracle over a table that points at an all-zero block."""
    kara = lib()
    spec = random_spec(530, G=4, hkv=2, W=64, B=16, D=128, n_seq=3, layers=1, len_lo=300, len_hi=1500)
    wl = synth.generate(spec)
    d = to_device(wl)
    q = synth.decode_queries(spec, 4)
    bt = wl.block_table.clone()
    bt[1, 3] = wl.num_blocks + 5
    got, st = run_decode(kara, d.k, d.v, spec.hq, 0, d.lengths, bt.cuda(), q.cuda())
    assert st == kara.EBADBLOCK
    zero = torch.zeros_like(wl.k[:, :1])
    kz, vz = torch.cat([wl.k, zero], 1), torch.cat([wl.v, zero], 1)
    bt_ref = wl.block_table.clone()
    bt_ref[1, 3] = wl.num_blocks
    s = wl.spec
    shape = oracle.make_shape(s.n_seq, s.layers, s.hq, s.hkv, s.d, s.block, s.W, s.B, s.K, s.R, s.lam,
                              wl.bt_stride, wl.num_blocks + 1)
    ref = oracle.decode_attention(shape, 0, q, kz, vz, bt_ref, wl.lengths)
    np.testing.assert_allclose(got, ref, atol=ATOL, rtol=RTOL)


def _decode_inputs(seed, n, hkv, G, D, nblk):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(1, nblk, hkv, 16, D, generator=g).to(torch.bfloat16)
    v = torch.randn(1, nblk, hkv, 16, D, generator=g).to(torch.bfloat16)
    q = torch.randn(n, G * hkv, D, generator=g).to(torch.bfloat16)
    return k, v, q


def test_decode_at_the_sequence_limit():
    """n = 65535 sequences (the largest batch a call takes), one block of 1..16
    keys each, block ids shuffled: every output against the oracle."""
    kara = lib()
    n, hkv, G, D = 65535, 1, 2, 64
    k, v, q = _decode_inputs(41, n, hkv, G, D, n)
    g = torch.Generator().manual_seed(42)
    lengths = torch.randint(1, 17, (n,), generator=g, dtype=torch.int32)
    bt = torch.randperm(n, generator=g).to(torch.int32).reshape(n, 1)
    got, st = run_decode(kara, k.cuda(), v.cuda(), G * hkv, 0, lengths.cuda(), bt.cuda(), q.cuda())
    assert st == 0
    sh = oracle.make_shape(n, 1, G * hkv, hkv, D, 16, 64, 16, 8, 16, 0.1, 1, n)
    ref = oracle.decode_attention(sh, 0, q, k, v, bt, lengths)
    np.testing.assert_allclose(got, ref, atol=ATOL, rtol=RTOL)


def test_decode_long_sequence_of_repeated_blocks():
    """One sequence of 4096 * 1024 keys (4096 splits) whose table cycles through
    the same 64 blocks: every key occurs equally often, so the exact result is
    the decode over those 1024 distinct keys once (oracle on a 64-block table)."""
    kara = lib()
    hkv, G, D, nblk = 2, 4, 128, 64
    splits = 4096
    L = splits * 1024
    k, v, q = _decode_inputs(43, 1, hkv, G, D, nblk)
    g = torch.Generator().manual_seed(44)
    cycle = torch.randperm(nblk, generator=g).to(torch.int32)
    bt = cycle.repeat(splits).reshape(1, splits * nblk)
    lengths = torch.tensor([L], dtype=torch.int32)
    got, st = run_decode(kara, k.cuda(), v.cuda(), G * hkv, 0, lengths.cuda(), bt.cuda(), q.cuda())
    assert st == 0
    sh = oracle.make_shape(1, 1, G * hkv, hkv, D, 16, 64, 16, 8, 16, 0.1, nblk, nblk)
    ref = oracle.decode_attention(sh, 0, q, k, v, cycle.reshape(1, nblk), torch.tensor([1024], dtype=torch.int32))
    np.testing.assert_allclose(got, ref, atol=ATOL, rtol=RTOL)
