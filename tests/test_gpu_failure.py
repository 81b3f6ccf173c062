"""Failure detection on the GPU without a fault, trap or hang.

With KARA_DEBUG_STALL=1 the kernels that stage data through shared memory
(the scorer's query strips, decode attention's K/V slices) issue no copies, so
their bounded waits run out on barriers that nothing will complete.  The call
reports KARA_ETIMEOUT through the error word, commits nothing, leaves every
live block as it was, and the next call on the same context is correct.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import random_spec
from _gpu import SCORE_RTOL, lib, rel_err, run_compress, to_device

pytestmark = pytest.mark.gpu


def test_stalled_scoring_times_out_and_commits_nothing(monkeypatch):
    kara = lib()
    spec = random_spec(901, G=4, hkv=2, W=512, B=64, D=128, n_seq=3, layers=2, len_lo=600, len_hi=1500)
    wl = synth.generate(spec)
    d = to_device(wl)
    k0, v0 = d.k.clone(), d.v.clone()

    monkeypatch.setenv("KARA_DEBUG_STALL", "1")
    out = run_compress(d)
    assert out["status"] == kara.ETIMEOUT
    assert np.array_equal(out["bt"], wl.block_table.numpy())       # the table is not rewritten
    assert np.array_equal(out["new_len"], wl.lengths.numpy())      # lengths stay
    fresh = set(wl.fresh.tolist())
    live = torch.tensor([b for b in range(wl.num_blocks) if b not in fresh], device="cuda")
    assert torch.equal(d.k[:, live], k0[:, live]) and torch.equal(d.v[:, live], v0[:, live])

    monkeypatch.delenv("KARA_DEBUG_STALL")
    out = run_compress(d)                                         # same context, normal call
    assert out["status"] == 0
    ref = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths)
    assert rel_err(out["scores"], ref).max() <= SCORE_RTOL


def test_stalled_decode_times_out(monkeypatch):
    kara = lib()
    spec = random_spec(902, G=4, hkv=2, W=64, B=16, D=128, n_seq=3, layers=1, len_lo=500, len_hi=2500)
    wl = synth.generate(spec)
    d = to_device(wl)
    q = synth.decode_queries(spec, 1).cuda()
    c = kara.cache(d.k, d.v, spec.hq)
    n, bts = d.block_table.shape
    ws = torch.empty(kara.kara_decode_workspace_size(c, n, bts), dtype=torch.uint8, device="cuda")

    def decode():
        out = torch.full((n, spec.hq, spec.d), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kara.kara_decode_attention(c, 0, d.lengths, d.block_table, q, out, ws, err)
        return out.cpu().numpy(), kara.kara_get_error(err)

    monkeypatch.setenv("KARA_DEBUG_STALL", "1")
    _, st = decode()
    assert st == kara.ETIMEOUT

    monkeypatch.delenv("KARA_DEBUG_STALL")
    got, st = decode()
    assert st == 0
    ref = oracle.decode_attention(oracle.shape_of(wl), 0, q.cpu(), wl.k, wl.v, wl.block_table, wl.lengths)
    np.testing.assert_allclose(got, ref, atol=2e-4, rtol=1e-3)
