"""GPU parity on K/V pools that are views with padded strides.

The scorer's tensor map, the decode kernel's tensor maps, the compaction and the
table commit all take the cache's layer, block and head strides.  Here the pools
are the [:, :num_blocks, :hkv] views of larger buffers whose padding holds a NaN
bit pattern: a kernel that addressed a row through the wrong stride would read
NaN into a result or write into the padding.  Scores, selection, the compacted
pools, the rewritten tables and decode attention over them are compared with
the oracle on the dense copies, and the padding must come back unchanged."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import random_spec
from _gpu import SCORE_RTOL, lib, rel_err

pytestmark = pytest.mark.gpu

NAN_BITS = 0x7FC0          # a quiet NaN in bf16
DEC_ATOL, DEC_RTOL = 2e-4, 1e-3


def padded_view(pool, extra_blocks, extra_heads):
    L, nb, hkv, bs, d = pool.shape
    big = torch.full((L, nb + extra_blocks, hkv + extra_heads, bs, d), NAN_BITS, dtype=torch.int16, device="cuda")
    view = big.view(torch.bfloat16)[:, :nb, :hkv]
    view.copy_(pool.to("cuda"))
    return big, view


def padding_intact(big, nb, hkv):
    return bool((big[:, nb:] == NAN_BITS).all()) and bool((big[:, :nb, hkv:] == NAN_BITS).all())


@pytest.mark.parametrize("D,G,W,B,K,R,extra_blocks,extra_heads", [
    (128, 5, 256, 32, 16, 60, 3, 1),
    (64, 2, 512, 64, 32, 120, 5, 2)])
def test_padded_pool_views(D, G, W, B, K, R, extra_blocks, extra_heads):
    kara = lib()
    spec = random_spec(930 + D + W, G=G, hkv=2, W=W, B=B, D=D, n_seq=3, layers=2, len_lo=W + 40,
                       len_hi=3 * W, K=K, R=R, plant="bernoulli")
    wl = synth.generate(spec)
    nb = wl.k.shape[1]
    kbig, k = padded_view(wl.k, extra_blocks, extra_heads)
    vbig, v = padded_view(wl.v, extra_blocks, extra_heads)
    assert k.stride(1) != spec.hkv * spec.block * D, "the view must not be dense"

    c = kara.cache(k, v, spec.hq)
    p = kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam)
    lengths = wl.lengths.cuda()
    bt = wl.block_table.cuda().contiguous()
    q = wl.q.cuda()
    b = kara.batch(lengths, bt, q)
    _, _, _, to = kara.kara_plan(p, spec.block, wl.lengths, wl.bt_stride)
    freed = torch.empty(max(to, 1), dtype=torch.int32, device="cuda")
    new_len = torch.empty(spec.n_seq, dtype=torch.int32, device="cuda")
    scores = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.C, dtype=torch.float32, device="cuda")
    kept = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.R, dtype=torch.int32, device="cuda")
    ws = torch.empty(kara.kara_workspace_size(c, p, spec.n_seq), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kara.kara_compress_batch(c, p, b, wl.fresh.cuda(), freed, new_len, ws, err, scores_out=scores, kept_out=kept)
    assert kara.kara_get_error(err) == 0

    sh = oracle.shape_of(wl)
    ref = oracle.scores(sh, wl.q, wl.k, wl.block_table, wl.lengths)
    got = scores.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert rel_err(got, ref).max() <= SCORE_RTOL
    _, kept_o = oracle.select_batch(got, spec.K, spec.R, spec.lam)
    assert np.array_equal(kept.cpu().numpy(), kept_o)
    st, k2, v2, bt2, fr2, nl2 = oracle.compact(sh, wl.k, wl.v, wl.block_table, wl.lengths, kept_o, wl.fresh)
    assert st == oracle.OK
    assert np.array_equal(bt.cpu().numpy(), bt2) and np.array_equal(new_len.cpu().numpy(), nl2)
    assert np.array_equal(freed.cpu().numpy()[:to], fr2)
    assert np.array_equal(k.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), k2)
    assert np.array_equal(v.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), v2)
    assert padding_intact(kbig, nb, spec.hkv) and padding_intact(vbig, nb, spec.hkv)

    # decode attention over the compacted views, through the rewritten tables
    dq = synth.decode_queries(spec, 3).cuda()
    dws = torch.empty(kara.kara_decode_workspace_size(c, spec.n_seq, wl.bt_stride), dtype=torch.uint8, device="cuda")
    for layer in range(spec.layers):
        out = torch.full((spec.n_seq, spec.hq, D), float("nan"), dtype=torch.float32, device="cuda")
        kara.kara_decode_attention(c, layer, new_len, bt, dq, out, dws, err)
        assert kara.kara_get_error(err) == 0
        dref = oracle.decode_attention(sh, layer, dq.cpu(), torch.from_numpy(k2.view(np.int16)),
                                       torch.from_numpy(v2.view(np.int16)), bt2, nl2)
        np.testing.assert_allclose(out.cpu().numpy(), dref, atol=DEC_ATOL, rtol=DEC_RTOL)
