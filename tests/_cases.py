"""Small hand-built and random cases for the oracle pins (CPU only)."""
import json
import os

import numpy as np
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16_bits_of(values) -> np.ndarray:
    """float values (exactly representable in bf16) -> uint16 bit patterns."""
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(np.asarray(values, dtype=np.float32))), "not bf16-exact"
    return t.view(torch.int16).numpy().view(np.uint16)


def golden_case(g):
    """Arrays for a hand-written score fixture."""
    sh = g["shape"]
    bt = np.asarray(g["block_table"], np.int32)
    nb = len(g["k_pool_rows"])
    rows = np.stack([np.asarray(g["k_pool_rows"][f"phys_block_{b}"], np.float32) for b in range(nb)])
    kpool = bf16_bits_of(rows).reshape(1, nb, 1, sh["block"], sh["d"])
    q = bf16_bits_of(np.asarray(g["q_rows"], np.float32)).reshape(1, 1, 1, sh["W"], sh["d"])
    shape = oracle.make_shape(sh["n_seq"], sh["layers"], sh["hq"], sh["hkv"], sh["d"], sh["block"],
                              sh["W"], sh["B"], sh["K"], sh["R"], sh["lam"], bt.shape[1], nb)
    return shape, q, kpool, bt, np.asarray(g["lengths"], np.int32)


def random_spec(seed, G=2, hkv=2, W=64, B=16, D=64, block=16, n_seq=2, layers=2, len_lo=None,
                len_hi=None, shuffled=True, plant="none", K=8, R=16):
    lo = len_lo if len_lo is not None else W
    hi = len_hi if len_hi is not None else W + 3 * block + 7
    return synth.Spec(f"rand{seed}", n_seq, layers, G * hkv, hkv, D, block, W, B, K, R, 0.1, lo, hi,
                      shuffled, plant, 0.05, seed)


def independent_colsum(wl, causal=False):
    """Column sums recomputed without the oracle: numpy gather + torch fp64 softmax
    (causal=True masks key j for window query i when j > i)."""
    s = wl.spec
    G = s.hq // s.hkv
    k = wl.k.float().double().numpy()
    q = wl.q.float().double()
    bt = wl.block_table.numpy()
    out = np.zeros((s.n_seq, s.layers, s.hkv, s.W))
    for si in range(s.n_seq):
        L = int(wl.lengths[si])
        pos = np.arange(L - s.W, L)
        blk = bt[si, pos // s.block]
        slot = pos % s.block
        for li in range(s.layers):
            for g in range(s.hkv):
                kw = torch.from_numpy(k[li, blk, g, slot, :])               # [W][D]
                qg = q[si, li, g * G:(g + 1) * G].reshape(-1, s.d)           # [G*W][D]
                lg = (qg @ kw.T) / np.sqrt(s.d)
                if causal:
                    i = torch.arange(G * s.W) % s.W
                    lg = lg.masked_fill(torch.arange(s.W)[None, :] > i[:, None], float("-inf"))
                p = torch.softmax(lg, dim=-1)
                out[si, li, g] = p.sum(dim=0).numpy()
    return out
