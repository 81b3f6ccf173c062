"""Periodic policy on the GPU: decode, compress a subset, decode on, compress again.

Each event goes through the host driver (decode_kv_cache_03_gb300.periodic)
and kara_compress_batch, and is checked against the oracle on a host copy of
the live cache: scores within tolerance, selection bit-exact on the GPU's
scores, and the pools, tables, lengths and freed ids bit-exact -- so the tables
the library rewrote are the ones the next event reads.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import SCORE_RTOL, lib, rel_err, to_device

pytestmark = pytest.mark.gpu


def test_consecutive_periods_match_oracle():
    lib()
    from decode_kv_cache_03_gb300 import Compressor
    from decode_kv_cache_03_gb300.periodic import BlockPool, PeriodicSchedule, append_tokens, compress_selected
    spec = synth.sweep_spec(5, 128).with_(layers=2, len_lo=300, len_hi=420, shuffled=True)
    wl = synth.generate(spec, extra_fresh_per_seq=24)
    d = to_device(wl)
    comp = Compressor(d.k, d.v, spec.hq, spec.W, spec.B, spec.K, spec.R, spec.lam)
    lengths = wl.lengths.tolist()
    stride = wl.bt_stride + 8
    table = torch.full((spec.n_seq, stride), -1, dtype=torch.int32)
    table[:, :wl.bt_stride] = wl.block_table
    pool = BlockPool(wl.fresh.tolist())
    sched = PeriodicSchedule(40, 0.5, spec.W, seed=5)
    gen = torch.Generator(device="cuda").manual_seed(11)
    events = 0
    for step in range(1, 121):
        before = list(lengths)
        append_tokens(lengths, table, pool, spec.block)
        # the new token of every sequence gets random K and V rows
        for s in range(spec.n_seq):
            x = before[s]
            blk, slot = int(table[s, x // spec.block]), x % spec.block
            d.k[:, blk, :, slot] = torch.randn(spec.layers, spec.hkv, spec.d, generator=gen, device="cuda").to(torch.bfloat16)
            d.v[:, blk, :, slot] = torch.randn(spec.layers, spec.hkv, spec.d, generator=gen, device="cuda").to(torch.bfloat16)
        if not sched.due(step):
            continue
        seqs = sched.choose(lengths)
        m = len(seqs)
        q = torch.randn(m, spec.layers, spec.hq, spec.W, spec.d, generator=gen, device="cuda").to(torch.bfloat16)
        sel_len = np.asarray([lengths[s] for s in seqs], np.int32)
        sel_bt = table[seqs].numpy().copy()
        kh = d.k.view(torch.int16).cpu().numpy().view(np.uint16)
        vh = d.v.view(torch.int16).cpu().numpy().view(np.uint16)
        nn, _ = oracle.plan(sel_len, spec.W, spec.B, spec.R, spec.block, stride)
        fresh_ids = np.asarray(pool.free[:int(nn.sum())], np.int32)
        scores = torch.empty(m, spec.layers, spec.hkv, spec.C, device="cuda")
        kept = torch.empty(m, spec.layers, spec.hkv, spec.R, dtype=torch.int32, device="cuda")
        freed, status = compress_selected(comp, seqs, lengths, table, q, pool, scores=scores, kept=kept)
        assert status == 0
        sh = oracle.make_shape(m, spec.layers, spec.hq, spec.hkv, spec.d, spec.block, spec.W, spec.B, spec.K,
                               spec.R, spec.lam, stride, wl.num_blocks)
        ref = oracle.scores(sh, q.cpu(), kh, sel_bt, sel_len)
        sc = scores.cpu().numpy()
        assert rel_err(sc, ref).max() <= SCORE_RTOL
        _, kept_o = oracle.select_batch(sc, spec.K, spec.R, spec.lam)
        assert np.array_equal(kept.cpu().numpy(), kept_o)
        st, k2, v2, bt2, fr2, nl2 = oracle.compact(sh, kh, vh, sel_bt, sel_len, kept_o, fresh_ids)
        assert st == oracle.OK
        assert np.array_equal(d.k.view(torch.int16).cpu().numpy().view(np.uint16), k2)
        assert np.array_equal(d.v.view(torch.int16).cpu().numpy().view(np.uint16), v2)
        assert np.array_equal(table[seqs].numpy(), bt2)
        assert [lengths[s] for s in seqs] == nl2.tolist()
        assert freed == fr2.tolist()
        events += 1
    assert events == 3
