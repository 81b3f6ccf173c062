"""GPU parity: the CUDA library through its C ABI against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import random_spec
from _gpu import SCORE_RTOL, lib, rel_err, run_compress, stable_windows, to_device

pytestmark = pytest.mark.gpu


def small(name, **kw):
    return synth.SPECS[name].with_(**kw)


E2E_CASES = {
    "tiny": synth.SPECS["tiny"],
    "qwen3_4b_small": small("qwen3_4b", n_seq=3, layers=2),
    "qwen3_14b_small": small("qwen3_14b", n_seq=2, layers=1, len_lo=2048, len_hi=4100),
    "llama_8b_small": small("llama_8b", n_seq=4, layers=2, len_lo=1024, len_hi=2100),
    "sweep_w128": synth.sweep_spec(4, 128).with_(layers=2),
    "sweep_w2048": synth.sweep_spec(1, 2048).with_(layers=1),
    "ragged_g3": random_spec(77, G=3, hkv=2, W=192, B=40, D=128, n_seq=3, layers=2, K=20, R=50,
                             len_lo=192, len_hi=400),
}


@pytest.mark.parametrize("case", list(E2E_CASES))
def test_compress_batch_matches_oracle(case):
    spec = E2E_CASES[case]
    wl = synth.generate(spec)
    out = run_compress(to_device(wl))
    assert out["status"] == 0
    sh = oracle.shape_of(wl)
    ref = oracle.scores(sh, wl.q, wl.k, wl.block_table, wl.lengths)
    # 1. scores within 1e-3 relative, element by element
    err = rel_err(out["scores"], ref)
    assert err.max() <= SCORE_RTOL, f"max rel err {err.max():.3e}"
    # 2. selection on the GPU's own scores is bit-exact
    cand_o, kept_o = oracle.select_batch(out["scores"], spec.K, spec.R, spec.lam)
    assert np.array_equal(out["cand"], cand_o)
    assert np.array_equal(out["kept"], kept_o)
    # 3. compaction, tables, freed ids and lengths bit-exact given the GPU's kept
    st, k2, v2, bt2, freed, new_len = oracle.compact(sh, wl.k, wl.v, wl.block_table, wl.lengths,
                                                     out["kept"], wl.fresh)
    assert st == oracle.OK
    assert np.array_equal(out["bt"], bt2)
    assert np.array_equal(out["freed"], freed)
    assert np.array_equal(out["new_len"], new_len)
    assert np.array_equal(out["k"], k2) and np.array_equal(out["v"], v2)
    # 4. end to end against the oracle's own selection, on tolerance-stable windows
    _, kept_ref = oracle.select_batch(ref, spec.K, spec.R, spec.lam)
    same = np.all(out["kept"] == kept_ref, axis=-1)
    stable = stable_windows(ref, spec.K, spec.R, spec.lam)
    assert np.all(same[stable]), f"{(~same[stable]).sum()} stable windows differ"
    assert same.mean() >= 0.9, f"exact-match rate {same.mean():.3f}"


@pytest.mark.parametrize("seed", range(6))
def test_select_bitexact_with_ties(seed):
    kara = lib()
    rng = np.random.default_rng(seed)
    W = int(rng.choice([64, 512, 1024, 2048]))
    B = int(rng.choice([0, 16, W // 8]))
    C = W - B
    K = int(rng.choice([1, 2, 8, min(C, 256), min(C, 1024)]))
    R = int(rng.choice([1, K, min(C, 89), C // 2, C]))
    nwin = 37
    if seed % 2:
        s = rng.choice(np.float32([0.5, 1.0, 1.0000001, 2.0, 0.0, -0.0]), size=(nwin, C))
    else:
        s = rng.exponential(size=(nwin, C)).astype(np.float32)
    sc = torch.from_numpy(s.astype(np.float32)).cuda()
    cand = torch.empty(nwin, K, dtype=torch.int32, device="cuda")
    kept = torch.empty(nwin, R, dtype=torch.int32, device="cuda")
    kara.kara_select(kara.params(W, B, K, R, 0.1), nwin, sc, cand, kept)
    torch.cuda.synchronize()
    c_o, k_o = oracle.select_batch(s, K, R, 0.1)
    assert np.array_equal(cand.cpu().numpy(), c_o)
    assert np.array_equal(kept.cpu().numpy(), k_o)


def test_select_stays_in_range_on_nan_scores():
    """NaN scores have no order to follow, but the result must still be a valid selection."""
    kara = lib()
    rng = np.random.default_rng(3)
    W, B, K, R, nwin = 1024, 128, 128, 268, 23
    C = W - B
    s = rng.random((nwin, C)).astype(np.float32)
    s[rng.random(s.shape) < 0.3] = np.nan
    s[0] = np.nan
    cand = torch.empty(nwin, K, dtype=torch.int32, device="cuda")
    kept = torch.empty(nwin, R, dtype=torch.int32, device="cuda")
    kara.kara_select(kara.params(W, B, K, R, 0.1), nwin, torch.from_numpy(s).cuda(), cand, kept)
    torch.cuda.synchronize()
    for arr, n in ((cand.cpu().numpy(), K), (kept.cpu().numpy(), R)):
        assert arr.shape[1] == n and np.all(np.diff(arr, axis=1) > 0) and arr.min() >= 0 and arr.max() < C


def test_score_alone_matches_oracle():
    kara = lib()
    spec = random_spec(5, G=4, hkv=2, W=256, B=32, D=128, n_seq=2, layers=2, len_lo=300, len_hi=700)
    wl = synth.generate(spec)
    d = to_device(wl)
    c = kara.cache(d.k, d.v, spec.hq)
    p = kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam)
    b = kara.batch(d.lengths, d.block_table, d.q)
    scores = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.C, dtype=torch.float32, device="cuda")
    ws = torch.empty(kara.kara_workspace_size(c, p, spec.n_seq), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kara.kara_score(c, p, b, scores, ws, err)
    assert kara.kara_get_error(err) == 0
    ref = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths)
    assert rel_err(scores.cpu().numpy(), ref).max() <= SCORE_RTOL


SCORE_SHAPES = [
    # (G, W, B, D): cluster sizes 1..8 (W up to 2048 on the single-pass kernel), partial
    # last key slice, partial last query strip, CTAs with 0, 1 or 2 compressible tiles,
    # both head dims
    (2, 64, 16, 64), (1, 64, 8, 128), (3, 192, 40, 128), (2, 256, 32, 128), (5, 320, 72, 64),
    (4, 512, 64, 128), (1, 640, 100, 128), (5, 1024, 128, 128), (8, 1024, 300, 64), (4, 2048, 256, 128),
    (2, 1600, 700, 128), (3, 1280, 200, 64), (2, 1536, 100, 128), (1, 1792, 300, 128),
]


@pytest.mark.parametrize("G,W,B,D", SCORE_SHAPES)
def test_score_shapes(G, W, B, D):
    kara = lib()
    spec = random_spec(500 + W + G, G=G, hkv=2, W=W, B=B, D=D, n_seq=2, layers=1, len_lo=W, len_hi=W + 40,
                       plant="bernoulli")
    wl = synth.generate(spec)
    d = to_device(wl)
    c = kara.cache(d.k, d.v, spec.hq)
    p = kara.params(spec.W, spec.B, 1, 1, spec.lam)
    b = kara.batch(d.lengths, d.block_table, d.q)
    scores = torch.full((spec.n_seq, spec.layers, spec.hkv, spec.C), -1.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(kara.kara_workspace_size(c, p, spec.n_seq), 1), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kara.kara_score(c, p, b, scores, ws, err)
    assert kara.kara_get_error(err) == 0
    ref = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths)
    e = rel_err(scores.cpu().numpy(), ref)
    assert e.max() <= SCORE_RTOL, f"max rel err {e.max():.3e} at {np.unravel_index(e.argmax(), e.shape)}"


@pytest.mark.parametrize("scale,W", [(60.0, 384), (-1e-3, 512)])
def test_windows_outside_the_single_pass_range_are_recomputed(scale, W):
    """The single-pass scorer exponentiates against the log-sum-exp of the same
    row position two strips earlier.  Here the query rows of the window's third
    strip are scaled so that reference is far off: by 60 (logits ~2^250 above
    it, the fp32 exponentials overflow) or by a tiny negative factor with the
    earlier strips' logits large (every term underflows).  Those windows must
    leave the single-pass arithmetic's range, be marked, and be recomputed
    exactly, so the scores still match the oracle."""
    kara = lib()
    spec = random_spec(931, G=1, hkv=2, W=W, B=32, D=128, n_seq=2, layers=1, len_lo=W, len_hi=W + 40)
    wl = synth.generate(spec)
    q = wl.q.float()
    if scale > 0:
        q[..., 256:, :] *= scale                   # strip 2 (rows 256..) of every window
    else:
        q[..., :256, :] *= 60.0                    # strips 0 and 1 large, strip 2 tiny
        q[..., 256:, :] *= -scale
    wl = synth.Workload(spec, q.to(torch.bfloat16), wl.k, wl.v, wl.lengths, wl.block_table, wl.fresh,
                        wl.prefix_pool, wl.fresh_base)
    d = to_device(wl)
    c = kara.cache(d.k, d.v, spec.hq)
    p = kara.params(spec.W, spec.B, 1, 1, spec.lam)
    b = kara.batch(d.lengths, d.block_table, d.q)
    scores = torch.full((spec.n_seq, spec.layers, spec.hkv, spec.C), -1.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(kara.kara_workspace_size(c, p, spec.n_seq), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kara.kara_score(c, p, b, scores, ws, err)
    assert kara.kara_get_error(err) == 0
    ref = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths)
    got = scores.cpu().numpy()
    assert np.all(np.isfinite(got))
    e = rel_err(got, ref)
    assert e.max() <= SCORE_RTOL, f"max rel err {e.max():.3e} at {np.unravel_index(e.argmax(), e.shape)}"


def test_compact_alone_with_oracle_kept():
    kara = lib()
    spec = random_spec(6, G=2, hkv=2, W=128, B=16, D=64, n_seq=3, layers=2, R=30, len_lo=128, len_hi=300)
    wl = synth.generate(spec)
    rng = np.random.default_rng(1)
    kept = np.sort(np.stack([rng.choice(spec.C, spec.R, replace=False)
                             for _ in range(spec.n_windows)]), axis=-1).astype(np.int32)
    kept = kept.reshape(spec.n_seq, spec.layers, spec.hkv, spec.R)
    d = to_device(wl)
    c = kara.cache(d.k, d.v, spec.hq)
    p = kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam)
    bt = d.block_table.clone()
    b = kara.batch(d.lengths, bt, d.q)
    _, _, tn, to = kara.kara_plan(p, 16, wl.lengths, wl.bt_stride)
    freed = torch.empty(to, dtype=torch.int32, device="cuda")
    new_len = torch.empty(spec.n_seq, dtype=torch.int32, device="cuda")
    ws = torch.empty(kara.kara_workspace_size(c, p, spec.n_seq), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kara.kara_compact(c, p, b, torch.from_numpy(kept).cuda(), d.fresh, freed, new_len, err, ws)
    assert kara.kara_get_error(err) == 0
    st, k2, v2, bt2, fr2, nl2 = oracle.compact(oracle.shape_of(wl), wl.k, wl.v, wl.block_table, wl.lengths,
                                              kept, wl.fresh)
    assert np.array_equal(bt.cpu().numpy(), bt2) and np.array_equal(freed.cpu().numpy(), fr2)
    assert np.array_equal(new_len.cpu().numpy(), nl2)
    assert np.array_equal(d.k.view(torch.int16).cpu().numpy().view(np.uint16), k2)
    assert np.array_equal(d.v.view(torch.int16).cpu().numpy().view(np.uint16), v2)


def _error_case(mutate):
    spec = random_spec(8, G=2, hkv=2, W=64, B=16, D=64, n_seq=3, layers=1, R=16)
    wl = synth.generate(spec)
    n_fresh = mutate(wl)
    d = to_device(wl)
    k0, v0, bt0 = d.k.clone(), d.v.clone(), d.block_table.clone()
    out = run_compress(d, n_fresh=n_fresh)
    return wl, out, k0, v0, bt0


def _assert_nothing_committed(wl, out, bt0):
    assert np.array_equal(out["bt"], bt0.cpu().numpy())
    assert np.array_equal(out["new_len"], wl.lengths.numpy())
    # old (non-fresh) blocks are never written
    fb = wl.fresh_base
    assert np.array_equal(out["k"][:, :fb], wl.k.view(torch.int16).numpy().view(np.uint16)[:, :fb])


def test_bad_block_id_is_reported_and_nothing_committed():
    def mutate(wl):
        L = int(wl.lengths[1])
        wl.block_table[1, (L - 1) // 16] = wl.num_blocks + 3
    wl, out, _, _, bt0 = _error_case(mutate)
    assert out["status"] == lib().EBADBLOCK
    _assert_nothing_committed(wl, out, bt0)


def test_short_fresh_list_is_reported_and_nothing_committed():
    wl, out, _, _, bt0 = _error_case(lambda wl: 1)
    assert out["status"] == lib().ENOBLOCKS
    _assert_nothing_committed(wl, out, bt0)


def test_short_sequence_is_reported_and_nothing_committed():
    def mutate(wl):
        wl.lengths[2] = 40
    spec = random_spec(8, G=2, hkv=2, W=64, B=16, D=64, n_seq=3, layers=1, R=16)
    wl = synth.generate(spec)
    mutate(wl)
    d = to_device(wl)
    kara = lib()
    # the host plan refuses it too
    with pytest.raises(kara.KaraError):
        kara.kara_plan(kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam), 16, wl.lengths, wl.bt_stride)
    bt0 = d.block_table.clone()
    s = spec
    c = kara.cache(d.k, d.v, s.hq)
    p = kara.params(s.W, s.B, s.K, s.R, s.lam)
    bt = d.block_table.clone()
    b = kara.batch(d.lengths, bt, d.q)
    freed = torch.full((64,), -7, dtype=torch.int32, device="cuda")
    new_len = torch.empty(s.n_seq, dtype=torch.int32, device="cuda")
    ws = torch.empty(kara.kara_workspace_size(c, p, s.n_seq), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kara.kara_compress_batch(c, p, b, d.fresh, freed, new_len, ws, err)
    assert kara.kara_get_error(err) == kara.EINVAL
    assert torch.equal(bt, bt0)
    assert torch.equal(new_len.cpu(), wl.lengths)
    assert torch.all(freed == -7)
