"""CUDA-graph capture of the step and of decode attention.

A serving loop captures its per-step work once and replays it.  Under capture
kara_compress_batch takes the one-pass sequence (no side streams), and decode
attention launches its merge kernel as a programmatic dependent of the split
kernel.  Each replay must produce the same bytes as eager calls on the same
inputs: scores, kept rows, the rewritten table, new lengths, freed ids, the
compacted pools, and the decode outputs of every layer."""
import numpy as np
import pytest
import torch

import synth
from _cases import random_spec
from _gpu import lib

pytestmark = pytest.mark.gpu


def _state(wl):
    return dict(k=wl.k.cuda(), v=wl.v.cuda(), bt=wl.block_table.cuda().contiguous(), lengths=wl.lengths.cuda(),
                q=wl.q.cuda(), fresh=wl.fresh.cuda())


def _outputs(kara, spec, st, to):
    return dict(freed=torch.full((max(to, 1),), -7, dtype=torch.int32, device="cuda"),
                new_len=torch.full((spec.n_seq,), -7, dtype=torch.int32, device="cuda"),
                scores=torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.C, dtype=torch.float32, device="cuda"),
                kept=torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.R, dtype=torch.int32, device="cuda"),
                err=torch.zeros(1, dtype=torch.int32, device="cuda"),
                dec=[torch.full((spec.n_seq, spec.hq, spec.d), float("nan"), device="cuda")
                     for _ in range(spec.layers)])


def _step(kara, spec, st, o, ws, dws, bt0, dq, restore):
    """One step as a serving loop runs it: (restore the table,) compress, then
    decode every layer over the new lengths and the rewritten table."""
    c = kara.cache(st["k"], st["v"], spec.hq)
    p = kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam)
    if restore:
        st["bt"].copy_(bt0)
    b = kara.batch(st["lengths"], st["bt"], st["q"])
    kara.kara_compress_batch(c, p, b, st["fresh"], o["freed"], o["new_len"], ws, o["err"],
                             scores_out=o["scores"], kept_out=o["kept"])
    for layer in range(spec.layers):
        kara.kara_decode_attention(c, layer, o["new_len"], st["bt"], dq, o["dec"][layer], dws, o["err"])


@pytest.mark.parametrize("W,D,G", [(256, 128, 4), (512, 64, 2)])
def test_graph_replay_matches_eager(W, D, G):
    kara = lib()
    spec = random_spec(950 + W + D, G=G, hkv=2, W=W, B=W // 8, D=D, n_seq=4, layers=2, len_lo=W + 100,
                       len_hi=4 * W, K=W // 16, R=W // 4, plant="bernoulli")
    wl = synth.generate(spec)
    c0 = kara.cache(wl.k, wl.v, spec.hq)
    p = kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam)
    _, _, _, to = kara.kara_plan(p, spec.block, wl.lengths, wl.bt_stride)
    ws_bytes = kara.kara_workspace_size(c0, p, spec.n_seq)
    dws_bytes = kara.kara_decode_workspace_size(c0, spec.n_seq, wl.bt_stride)
    dq = synth.decode_queries(spec, 5).cuda()
    bt0 = wl.block_table.cuda().contiguous()

    # eager
    se = _state(wl)
    oe = _outputs(kara, spec, se, to)
    _step(kara, spec, se, oe, torch.empty(ws_bytes, dtype=torch.uint8, device="cuda"),
          torch.empty(dws_bytes, dtype=torch.uint8, device="cuda"), bt0, dq, restore=False)
    torch.cuda.synchronize()
    assert kara.kara_get_error(oe["err"]) == 0

    # captured once, replayed twice (the captured copy restores the table first)
    sg = _state(wl)
    og = _outputs(kara, spec, sg, to)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    dws = torch.empty(dws_bytes, dtype=torch.uint8, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(kara, spec, sg, og, ws, dws, bt0, dq, restore=True)
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        assert kara.kara_get_error(og["err"]) == 0
        for key in ("freed", "new_len", "scores", "kept"):
            assert torch.equal(og[key], oe[key]), key
        assert torch.equal(sg["bt"], se["bt"])
        for pool in ("k", "v"):
            assert torch.equal(sg[pool].view(torch.int16), se[pool].view(torch.int16)), pool
        for layer in range(spec.layers):
            assert torch.equal(og["dec"][layer], oe["dec"][layer]), layer
            assert bool(torch.isfinite(og["dec"][layer]).all())
