"""Helpers for the GPU parity tests: run the library through its C ABI and the
oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle
import synth

SCORE_RTOL = 1e-3          # scores: fp32 accumulation from bf16 vs the fp64 oracle


def lib():
    from decode_kv_cache_03_gb300 import build
    build.build()
    from decode_kv_cache_03_gb300 import kara
    return kara


def to_device(wl: synth.Workload) -> synth.Workload:
    d = "cuda"
    return synth.Workload(wl.spec, wl.q.to(d), wl.k.to(d), wl.v.to(d), wl.lengths.to(d),
                          wl.block_table.to(d).contiguous(), wl.fresh.to(d), wl.prefix_pool, wl.fresh_base)


def run_compress(wl_dev: synth.Workload, n_fresh=None, score_mode=0, select_mode=0, chunk=0):
    """kara_compress_batch on device data; returns host copies of every output."""
    kara = lib()
    s = wl_dev.spec
    c = kara.cache(wl_dev.k, wl_dev.v, s.hq)
    p = kara.params(s.W, s.B, s.K, s.R, s.lam, score_mode, select_mode, chunk)
    bt = wl_dev.block_table.clone()
    b = kara.batch(wl_dev.lengths, bt, wl_dev.q)
    nn, no, tn, to = kara.kara_plan(p, s.block, wl_dev.lengths.cpu(), wl_dev.bt_stride)
    fresh = wl_dev.fresh if n_fresh is None else wl_dev.fresh[:n_fresh]
    freed = torch.full((max(to, 1),), -7, dtype=torch.int32, device="cuda")
    new_len = torch.full((s.n_seq,), -7, dtype=torch.int32, device="cuda")
    scores = torch.empty(s.n_seq, s.layers, s.hkv, s.C, dtype=torch.float32, device="cuda")
    cand = torch.empty(s.n_seq, s.layers, s.hkv, s.K, dtype=torch.int32, device="cuda")
    kept = torch.empty(s.n_seq, s.layers, s.hkv, s.R, dtype=torch.int32, device="cuda")
    ws = torch.empty(kara.kara_workspace_size(c, p, s.n_seq), dtype=torch.uint8, device="cuda")
    err = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    kara.kara_compress_batch(c, p, b, fresh, freed, new_len, ws, err, scores, cand, kept)
    status = kara.kara_get_error(err)
    torch.cuda.synchronize()
    return dict(status=status, scores=scores.cpu().numpy(), cand=cand.cpu().numpy(), kept=kept.cpu().numpy(),
                bt=bt.cpu().numpy(), freed=freed.cpu().numpy()[:to], new_len=new_len.cpu().numpy(),
                k=wl_dev.k.view(torch.int16).cpu().numpy().view(np.uint16),
                v=wl_dev.v.view(torch.int16).cpu().numpy().view(np.uint16))


def stable_windows(scores_ref, K, R, lam, trials=6, eps=1e-4, seed=0):
    """Windows whose oracle selection does not move under random relative
    perturbations of eps (100x the fp32 error seen in practice)."""
    rng = np.random.default_rng(seed)
    C = scores_ref.shape[-1]
    flat = scores_ref.reshape(-1, C)
    base = oracle.select_batch(flat, K, R, lam)[1]
    ok = np.ones(flat.shape[0], bool)
    for _ in range(trials):
        pert = (flat * (1 + eps * rng.uniform(-1, 1, flat.shape))).astype(np.float32)
        ok &= np.all(oracle.select_batch(pert, K, R, lam)[1] == base, axis=-1)
    return ok.reshape(scores_ref.shape[:-1])


def rel_err(a, b):
    return np.abs(a.astype(np.float64) - b.astype(np.float64)) / np.maximum(np.abs(b.astype(np.float64)), 1e-30)
