"""kara_compress_batch in groups of sequences: the selection, kept-row check and
copy of one group run on a second stream while the next group is scored.

The groups run the same kernels on the same windows as the unpipelined
sequence, and a window's scores depend on that window only, so every output
(scores, candidates, kept rows, pools, tables, freed ids, new lengths) must be
the same bytes, and match the oracle.  The fresh-id
check still covers the whole batch before any block is written, and the
tables are committed only after every group, only without an error.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import random_spec
from _gpu import SCORE_RTOL, lib, rel_err, run_compress, to_device

pytestmark = pytest.mark.gpu


def small(name, **kw):
    return synth.SPECS[name].with_(**kw)


CASES = {
    # single-pass scorer, 4-CTA clusters
    "qwen3_14b_3seq": (small("qwen3_14b", n_seq=3, layers=1, len_lo=2048, len_hi=4100), 3),
    # single-pass scorer, 2-CTA clusters
    "qwen3_4b_3seq": (small("qwen3_4b", n_seq=3, layers=2), 2),
    # single-pass scorer, one CTA per window
    "llama_8b_4seq": (small("llama_8b", n_seq=4, layers=2, len_lo=1024, len_hi=2100), 4),
    # uneven groups (1, 1, 2 sequences)
    "sweep_w128": (synth.sweep_spec(4, 128).with_(layers=2), 3),
    # 8 key slices per window (8-CTA clusters, one key buffer)
    "sweep_w2048": (synth.sweep_spec(2, 2048).with_(layers=1), 2),
    "ragged_g3": (random_spec(77, G=3, hkv=2, W=192, B=40, D=128, n_seq=3, layers=2, K=20, R=50,
                              len_lo=192, len_hi=400), 3),
}


def _groups(kara, d):
    s = d.spec
    c = kara.cache(d.k, d.v, s.hq)
    p = kara.params(s.W, s.B, s.K, s.R, s.lam)
    b = kara.batch(d.lengths, d.block_table, d.q)
    return kara.kara_batch_groups(c, p, b)


@pytest.mark.parametrize("case", list(CASES))
def test_groups_give_the_same_bytes_as_one_pass(case, monkeypatch):
    spec, m = CASES[case]
    kara = lib()
    wl = synth.generate(spec)
    out = {}
    for groups in (1, m):
        monkeypatch.setenv("KARA_BATCH_GROUPS", str(groups))
        d = to_device(wl)
        assert _groups(kara, d) == groups
        out[groups] = run_compress(d)
    a, b = out[1], out[m]
    assert a["status"] == 0 and b["status"] == 0
    for key in ("scores", "cand", "kept", "bt", "freed", "new_len", "k", "v"):
        assert np.array_equal(a[key], b[key]), key
    # and the oracle, as for the unpipelined call
    sh = oracle.shape_of(wl)
    ref = oracle.scores(sh, wl.q, wl.k, wl.block_table, wl.lengths)
    assert rel_err(b["scores"], ref).max() <= SCORE_RTOL
    cand_o, kept_o = oracle.select_batch(b["scores"], spec.K, spec.R, spec.lam)
    assert np.array_equal(b["cand"], cand_o) and np.array_equal(b["kept"], kept_o)
    st, k2, v2, bt2, freed, new_len = oracle.compact(sh, wl.k, wl.v, wl.block_table, wl.lengths, b["kept"],
                                                     wl.fresh)
    assert st == oracle.OK
    assert np.array_equal(b["bt"], bt2) and np.array_equal(b["freed"], freed)
    assert np.array_equal(b["new_len"], new_len)
    assert np.array_equal(b["k"], k2) and np.array_equal(b["v"], v2)


def _spec():
    return random_spec(8, G=2, hkv=2, W=64, B=16, D=64, n_seq=3, layers=2, R=16)


def test_bad_block_in_the_last_group_commits_nothing(monkeypatch):
    """A block id outside the pool in the last group's sequence: reported, no
    table or length changes, no live block written (earlier groups may have
    filled fresh blocks)."""
    monkeypatch.setenv("KARA_BATCH_GROUPS", "3")
    wl = synth.generate(_spec())
    L = int(wl.lengths[2])
    wl.block_table[2, (L - 1) // 16] = wl.num_blocks + 3
    d = to_device(wl)
    assert _groups(lib(), d) == 3
    out = run_compress(d)
    assert out["status"] == lib().EBADBLOCK
    assert np.array_equal(out["bt"], wl.block_table.numpy())
    assert np.array_equal(out["new_len"], wl.lengths.numpy())
    fb = wl.fresh_base
    assert np.array_equal(out["k"][:, :fb], wl.k.view(torch.int16).numpy().view(np.uint16)[:, :fb])
    assert np.array_equal(out["v"][:, :fb], wl.v.view(torch.int16).numpy().view(np.uint16)[:, :fb])


def test_duplicate_fresh_id_writes_no_block_in_any_group(monkeypatch):
    """The fresh-id check covers the whole batch before the first group's copy."""
    monkeypatch.setenv("KARA_BATCH_GROUPS", "3")
    wl = synth.generate(_spec())
    nn, _ = oracle.plan(wl.lengths, wl.spec.W, wl.spec.B, wl.spec.R, wl.spec.block, wl.bt_stride)
    used = int(nn.sum())
    fresh = wl.fresh.clone()
    fresh[used - 1] = fresh[0]               # the last group's last fresh id repeats the first group's
    wl = synth.Workload(wl.spec, wl.q, wl.k, wl.v, wl.lengths, wl.block_table, fresh, wl.prefix_pool,
                        wl.fresh_base)
    want = oracle.compact(oracle.shape_of(wl), wl.k, wl.v, wl.block_table, wl.lengths,
                          np.tile(np.arange(wl.spec.R, dtype=np.int32),
                                  (wl.spec.n_seq, wl.spec.layers, wl.spec.hkv, 1)), fresh)[0]
    assert want == oracle.EDUPBLOCK
    d = to_device(wl)
    k0, v0 = d.k.clone(), d.v.clone()
    out = run_compress(d)
    assert out["status"] == lib().EDUPBLOCK
    assert np.array_equal(out["bt"], wl.block_table.numpy())
    assert np.array_equal(out["new_len"], wl.lengths.numpy())
    assert torch.equal(d.k.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(d.v.view(torch.int16), v0.view(torch.int16))


@pytest.mark.parametrize("W,layers", [(1024, 3), (2048, 2)])
def test_scores_depend_on_their_own_window_only(W, layers):
    """A window scored in a batch where each cluster of the persistent scorer
    walks several windows gets the same bits as when its sequence is scored
    alone."""
    kara = lib()
    spec = (synth.SPECS["qwen3_14b"].with_(n_seq=4, layers=layers, len_lo=2048, len_hi=4100) if W == 1024
            else synth.sweep_spec(4, 2048).with_(layers=layers))
    wl = synth.generate(spec)
    d = to_device(wl)

    def scores_of(lengths, bt, q, n):
        c = kara.cache(d.k, d.v, spec.hq)
        p = kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam)
        b = kara.batch(lengths, bt, q)
        out = torch.empty(n, spec.layers, spec.hkv, spec.C, dtype=torch.float32, device="cuda")
        ws = torch.empty(kara.kara_workspace_size(c, p, n), dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kara.kara_score(c, p, b, out, ws, err)
        assert kara.kara_get_error(err) == 0
        return out.cpu().numpy()

    every = scores_of(d.lengths, d.block_table, d.q, spec.n_seq)
    for s in (1, spec.n_seq - 1):
        alone = scores_of(d.lengths[s:s + 1].contiguous(), d.block_table[s:s + 1].contiguous(),
                          d.q[s:s + 1].contiguous(), 1)
        assert np.array_equal(alone[0].view(np.uint32), every[s].view(np.uint32)), s

