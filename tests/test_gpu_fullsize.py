"""Full-size workloads on the GPU, in the launch configuration the benchmark times.

The whole batch goes through one kara_compress_batch call (and its window-query
ring through one kara_compact_queries call); on the Qwen3-14B shape that call
runs in groups of sequences, the selection and copy of one group under the
scoring of the next.  A few windows,
sampled by a seeded generator, are recomputed by the oracle one by one from a
host copy of their inputs taken before the call; every window and every
sequence is also checked for properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import SCORE_RTOL, lib, rel_err

pytestmark = pytest.mark.gpu


def _sample(spec, seed, n_seq_sample=3):
    rng = np.random.default_rng(seed)
    seqs = sorted(rng.choice(spec.n_seq, size=min(n_seq_sample, spec.n_seq), replace=False).tolist())
    layer = int(rng.integers(spec.layers))
    return seqs, layer


@pytest.mark.parametrize("name", ["qwen3_14b", "qwen3_4b", "llama_8b"])
def test_full_batch(name):
    kara = lib()
    spec = synth.SPECS[name]
    wl = synth.generate(spec, device="cuda")           # same generator and layout as the benchmark
    seqs, layer = _sample(spec, 17)
    sub = synth.host_subset(wl, seqs)                  # inputs of the sampled windows, before the call
    bt_before = wl.block_table.cpu().numpy().copy()
    lengths = wl.lengths.cpu().numpy()

    c = kara.cache(wl.k, wl.v, spec.hq)
    p = kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam)
    b = kara.batch(wl.lengths, wl.block_table, wl.q)
    nn, no, tn, to = kara.kara_plan(p, spec.block, wl.lengths.cpu(), wl.bt_stride)
    freed = torch.full((to,), -7, dtype=torch.int32, device="cuda")
    new_len = torch.empty(spec.n_seq, dtype=torch.int32, device="cuda")
    scores = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.C, dtype=torch.float32, device="cuda")
    cand = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.K, dtype=torch.int32, device="cuda")
    kept = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.R, dtype=torch.int32, device="cuda")
    ws = torch.empty(kara.kara_workspace_size(c, p, spec.n_seq), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    groups = kara.kara_batch_groups(c, p, b)
    if name == "qwen3_14b":
        assert groups > 1      # the scorer's 36 clusters of 4 leave 8 of the 152 SMs idle
    kara.kara_compress_batch(c, p, b, wl.fresh, freed, new_len, ws, err, scores, cand, kept)
    assert kara.kara_get_error(err) == 0

    sc = scores.cpu().numpy()
    kp = kept.cpu().numpy()
    cd = cand.cpu().numpy()
    G = spec.hq // spec.hkv
    # --- properties of every window ---------------------------------------------
    assert np.all(np.isfinite(sc)) and np.all(sc > 0)
    assert np.all(sc.astype(np.float64).sum(-1) <= G * spec.W * (1 + 1e-5))
    assert np.all(np.diff(kp, axis=-1) > 0) and kp.min() >= 0 and kp.max() < spec.C
    assert np.all(np.diff(cd, axis=-1) > 0) and cd.min() >= 0 and cd.max() < spec.C
    # --- every sequence: lengths, tables and freed ids are exact ------------------
    rn, ro = oracle.plan(lengths, spec.W, spec.B, spec.R, spec.block, wl.bt_stride)
    bt_after = wl.block_table.cpu().numpy()
    fresh = wl.fresh.cpu().numpy()
    fr = freed.cpu().numpy()
    assert np.array_equal(new_len.cpu().numpy(), lengths - spec.C + spec.R)
    on = np.concatenate([[0], np.cumsum(rn)])
    oo = np.concatenate([[0], np.cumsum(ro)])
    for s in range(spec.n_seq):
        p0 = (int(lengths[s]) - spec.W) // spec.block
        nb_old = (int(lengths[s]) + spec.block - 1) // spec.block
        assert np.array_equal(bt_after[s, :p0], bt_before[s, :p0])
        assert np.array_equal(bt_after[s, p0:p0 + rn[s]], fresh[on[s]:on[s + 1]])
        assert np.all(bt_after[s, p0 + rn[s]:nb_old] == -1)
        assert np.array_equal(fr[oo[s]:oo[s + 1]], bt_before[s, p0:nb_old])
    # --- sampled windows against the oracle, one by one --------------------------
    ss = sub.spec.with_(layers=1)
    q1 = sub.q[:, layer:layer + 1].contiguous()
    k1 = sub.k[layer:layer + 1].contiguous()
    v1 = sub.v[layer:layer + 1].contiguous()
    sh = oracle.make_shape(ss.n_seq, 1, ss.hq, ss.hkv, ss.d, ss.block, ss.W, ss.B, ss.K, ss.R, ss.lam,
                           sub.bt_stride, sub.num_blocks)
    ref = oracle.scores(sh, q1, k1, sub.block_table, sub.lengths)
    got = sc[seqs][:, layer:layer + 1]
    assert rel_err(got, ref).max() <= SCORE_RTOL
    c_o, k_o = oracle.select_batch(got, spec.K, spec.R, spec.lam)
    assert np.array_equal(cd[seqs][:, layer:layer + 1], c_o)
    assert np.array_equal(kp[seqs][:, layer:layer + 1], k_o)
    # compacted rows of the sampled windows equal the oracle's compaction of them
    st, k2, v2, bt2, _, nl2 = oracle.compact(sh, k1, v1, sub.block_table, sub.lengths, k_o, sub.fresh)
    assert st == oracle.OK
    kd = wl.k[layer].view(torch.int16)
    vd = wl.v[layer].view(torch.int16)
    for i, s in enumerate(seqs):
        p0 = (int(lengths[s]) - spec.W) // spec.block
        xs = np.arange(p0 * spec.block, int(nl2[i]))
        bg = torch.from_numpy(bt_after[s, xs // spec.block].astype(np.int64)).cuda()
        slot = torch.from_numpy(xs % spec.block).cuda()
        bo, so = bt2[i, xs // spec.block], xs % spec.block
        assert np.array_equal(kd[bg, :, slot].cpu().numpy().view(np.uint16), k2[0, bo, :, so])
        assert np.array_equal(vd[bg, :, slot].cpu().numpy().view(np.uint16), v2[0, bo, :, so])
    # --- the window queries kept as a ring, compacted with K and V over the whole
    # batch (as `bench.py --q-ring` runs it): the sampled sequences' rings, all
    # layers and heads, equal the oracle's compaction of their host copies
    kara.kara_compact_queries(c, p, b, kept, err)
    assert kara.kara_get_error(err) == 0
    ref_ring = oracle.compact_queries(oracle.shape_of(sub), sub.q, sub.lengths, kp[seqs])
    got_ring = wl.q[seqs].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_ring, ref_ring)


@pytest.mark.parametrize("name", ["qwen3_14b", "llama_8b"])
def test_full_layer_decode(name):
    """Decode attention over a whole layer of the workload, as `bench.py --decode`
    launches it; every output is finite and the outputs of a few sampled
    sequences equal the oracle's, recomputed from host copies of their blocks."""
    kara = lib()
    spec = synth.SPECS[name].with_(layers=1)
    wl = synth.generate(spec, device="cuda", alias_prefix=False, with_q=False)
    q = synth.decode_queries(spec, 0, device="cuda")
    c = kara.cache(wl.k, wl.v, spec.hq)
    n, bts = wl.block_table.shape
    ws = torch.empty(kara.kara_decode_workspace_size(c, n, bts), dtype=torch.uint8, device="cuda")
    out = torch.full((n, spec.hq, spec.d), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kara.kara_decode_attention(c, 0, wl.lengths, wl.block_table, q, out, ws, err)
    assert kara.kara_get_error(err) == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))

    seqs, _ = _sample(spec, 23)
    bt = wl.block_table[seqs].cpu()
    lens = wl.lengths[seqs].cpu()
    nblk = [(int(L) + spec.block - 1) // spec.block for L in lens]
    ids = sorted({int(bt[i, t]) for i in range(len(seqs)) for t in range(nblk[i])})
    remap = {b: j for j, b in enumerate(ids)}
    bt2 = torch.full_like(bt, -1)
    for i in range(len(seqs)):
        bt2[i, :nblk[i]] = torch.tensor([remap[int(b)] for b in bt[i, :nblk[i]]], dtype=torch.int32)
    idx = torch.tensor(ids, dtype=torch.int64, device="cuda")
    k2, v2 = wl.k[:, idx].cpu().contiguous(), wl.v[:, idx].cpu().contiguous()
    shape = oracle.make_shape(len(seqs), 1, spec.hq, spec.hkv, spec.d, spec.block, spec.W, spec.B, spec.K,
                              spec.R, spec.lam, bts, len(ids))
    ref = oracle.decode_attention(shape, 0, q[seqs].cpu(), k2, v2, bt2, lens)
    np.testing.assert_allclose(got[seqs], ref, atol=2e-4, rtol=1e-3)
