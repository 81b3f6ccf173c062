"""GPU parity of the ablation variants: causal window scores and the two
selection modes that replace Token2Chunk, each against the oracle on the same
seeded inputs (scores within SCORE_RTOL, selection and compaction bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import random_spec
from _gpu import SCORE_RTOL, lib, rel_err, run_compress, to_device

pytestmark = pytest.mark.gpu

CAUSAL_SHAPES = [
    # (G, W, B, D): a 64-wide window (strips span two heads), W = 64 mod 128 with
    # one and two key slices, full-size windows of 4 and 8 slices, both head dims
    (2, 64, 16, 64), (3, 192, 40, 128), (5, 320, 72, 64), (4, 512, 64, 128), (5, 1024, 128, 128),
    (4, 2048, 256, 128),
]


@pytest.mark.parametrize("G,W,B,D", CAUSAL_SHAPES)
def test_causal_scores_match_oracle(G, W, B, D):
    kara = lib()
    spec = random_spec(200 + W + G, G=G, hkv=2, W=W, B=B, D=D, n_seq=2, layers=1, len_lo=W, len_hi=W + 80,
                       plant="bernoulli")
    wl = synth.generate(spec)
    d = to_device(wl)
    c = kara.cache(d.k, d.v, spec.hq)
    b = kara.batch(d.lengths, d.block_table, d.q)
    out = {}
    for mode in (kara.SCORE_CAUSAL, kara.SCORE_BIDIRECTIONAL):
        p = kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam, score_mode=mode)
        scores = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.C, dtype=torch.float32, device="cuda")
        ws = torch.empty(max(1, kara.kara_workspace_size(c, p, spec.n_seq)), dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kara.kara_score(c, p, b, scores, ws, err)
        assert kara.kara_get_error(err) == 0
        out[mode] = scores.cpu().numpy()
    ref = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths, causal=True)
    assert rel_err(out[kara.SCORE_CAUSAL], ref).max() <= SCORE_RTOL
    assert not np.allclose(out[kara.SCORE_CAUSAL], out[kara.SCORE_BIDIRECTIONAL], rtol=1e-2)


@pytest.mark.parametrize("mode,chunk", [(1, 0), (2, 1), (2, 7), (2, 16), (2, -1)])
@pytest.mark.parametrize("seed", range(3))
def test_select_modes_bitexact(mode, chunk, seed):
    kara = lib()
    rng = np.random.default_rng(300 + seed)
    W = int(rng.choice([64, 512, 1024, 2048]))
    B = int(rng.choice([0, 16, W // 8]))
    C = W - B
    K = int(rng.choice([1, 8, min(C, 128)]))
    R = int(rng.choice([1, min(C, 89), C // 2, C]))
    ch = C if chunk == -1 else chunk
    nwin = 29
    if seed % 2:
        s = rng.choice(np.float32([0.5, 1.0, 1.0000001, 2.0, 0.0, -0.0]), size=(nwin, C))
    else:
        s = rng.exponential(size=(nwin, C)).astype(np.float32)
    cand = torch.empty(nwin, K, dtype=torch.int32, device="cuda")
    kept = torch.empty(nwin, R, dtype=torch.int32, device="cuda")
    p = kara.params(W, B, K, R, 0.1, select_mode=mode, chunk=ch)
    kara.kara_select(p, nwin, torch.from_numpy(s).cuda(), cand, kept)
    torch.cuda.synchronize()
    c_o, k_o = oracle.select_mode_batch(s, K, R, 0.1, mode, ch)
    assert np.array_equal(cand.cpu().numpy(), c_o)
    assert np.array_equal(kept.cpu().numpy(), k_o)


@pytest.mark.parametrize("score_mode,select_mode,chunk", [(1, 0, 0), (0, 1, 0), (0, 2, 8), (1, 2, 16)])
def test_compress_batch_with_modes(score_mode, select_mode, chunk):
    """The whole step under a variant: scores within tolerance of the oracle,
    selection bit-exact on the GPU's scores, K/V bytes and tables bit-exact."""
    spec = random_spec(400 + 4 * score_mode + select_mode, G=4, hkv=2, W=256, B=32, D=128, n_seq=3, layers=2,
                       len_lo=300, len_hi=700, plant="bernoulli", K=16, R=60)
    wl = synth.generate(spec)
    out = run_compress(to_device(wl), score_mode=score_mode, select_mode=select_mode, chunk=chunk)
    assert out["status"] == 0
    ref = oracle.scores(oracle.shape_of(wl), wl.q, wl.k, wl.block_table, wl.lengths, causal=bool(score_mode))
    assert rel_err(out["scores"], ref).max() <= SCORE_RTOL
    c_o, k_o = oracle.select_mode_batch(out["scores"], spec.K, spec.R, spec.lam, select_mode, chunk)
    assert np.array_equal(out["cand"], c_o)
    assert np.array_equal(out["kept"], k_o)
    kh = wl.k.view(torch.int16).numpy().view(np.uint16)
    vh = wl.v.view(torch.int16).numpy().view(np.uint16)
    st, k2, v2, bt2, fr2, nl2 = oracle.compact(oracle.shape_of(wl), kh, vh, wl.block_table, wl.lengths, k_o,
                                               wl.fresh)
    assert st == oracle.OK
    assert np.array_equal(out["k"], k2) and np.array_equal(out["v"], v2)
    assert np.array_equal(out["bt"], bt2) and np.array_equal(out["freed"], fr2)
    assert np.array_equal(out["new_len"], nl2)
