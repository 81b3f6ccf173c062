"""The C-ABI library loads and exports what include/kara.h declares (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from decode_kv_cache_03_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kara():
    kbuild.build()
    from decode_kv_cache_03_gb300 import kara as k
    return k


def declared_functions():
    names = set()
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(kara_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(kara):
    lib = ctypes.CDLL(kara.LIB_PATH)
    names = declared_functions()
    assert {"kara_score", "kara_select", "kara_compact", "kara_compress_batch", "kara_plan"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(kara.EXPORTED) <= names


def test_status_strings(kara):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert kara.status_string(code).startswith("KARA_")
    assert kara.version() == 1


@pytest.mark.parametrize("seed", range(5))
def test_host_plan_matches_oracle_plan(kara, seed):
    rng = np.random.default_rng(seed)
    W = int(rng.choice([64, 128, 512, 1024]))
    B = int(rng.integers(0, W))
    R = int(rng.integers(1, W - B + 1))
    K = 1
    lengths = rng.integers(W, W + 3000, size=50).astype(np.int32)
    bt_stride = int((lengths.max() + 15) // 16)
    nn, no, tn, to = kara.kara_plan(kara.params(W, B, K, R, 0.1), 16, torch.from_numpy(lengths), bt_stride)
    rn, ro = oracle.plan(lengths, W, B, R, 16, bt_stride)
    assert nn.numpy().tolist() == rn.tolist() and no.numpy().tolist() == ro.tolist()
    assert tn == int(rn.sum()) and to == int(ro.sum())


def test_host_plan_rejects(kara):
    p = kara.params(64, 16, 8, 16, 0.1)
    with pytest.raises(kara.KaraError) as e:
        kara.kara_plan(p, 16, torch.tensor([63], dtype=torch.int32), 10)
    assert e.value.status == kara.EINVAL
    with pytest.raises(kara.KaraError) as e:
        kara.kara_plan(kara.params(96, 16, 8, 16, 0.1), 16, torch.tensor([200], dtype=torch.int32), 20)
    assert e.value.status == kara.EUNSUPPORTED


def fake_cache(kara, **kw):
    c = kara.Cache(16, 16, 8 * 16 * 64 * 2, 2 * 16 * 64, 16 * 64, 1, 8, 2, 4, 64, 16)
    for k_, v_ in kw.items():
        setattr(c, k_, v_)
    return c


def test_argument_checks_happen_before_any_device_work(kara):
    """Invalid shapes are refused on the host with a status; nothing is launched."""
    p = kara.params(64, 16, 8, 16, 0.1)
    b = kara.Batch(1, 16, 16, 16, 16)
    ws = ctypes.c_void_p(16)
    cases = [
        (fake_cache(kara, head_dim=96), p, kara.EUNSUPPORTED),
        (fake_cache(kara, block_size=8), p, kara.EUNSUPPORTED),
        (fake_cache(kara, num_q_heads=3), p, kara.EINVAL),
        (fake_cache(kara, num_q_heads=2 * 9), p, kara.EUNSUPPORTED),
        (fake_cache(kara, k=None), p, kara.EINVAL),
        (fake_cache(kara, k=18), p, kara.EINVAL),
        (fake_cache(kara), kara.params(64, 64, 8, 16, 0.1), kara.EINVAL),
        (fake_cache(kara), kara.params(64, 16, 49, 16, 0.1), kara.EINVAL),
        (fake_cache(kara), kara.params(64, 16, 8, 49, 0.1), kara.EINVAL),
        (fake_cache(kara), kara.params(64, 16, 8, 0, 0.1), kara.EINVAL),
        (fake_cache(kara), kara.params(4096, 16, 8, 16, 0.1), kara.EUNSUPPORTED),
        (fake_cache(kara), kara.params(64, 16, 8, 16, 0.1, score_mode=2), kara.EINVAL),
        (fake_cache(kara), kara.params(64, 16, 8, 16, 0.1, select_mode=3), kara.EINVAL),
        (fake_cache(kara), kara.params(64, 16, 8, 16, 0.1, select_mode=2, chunk=0), kara.EINVAL),
        (fake_cache(kara), kara.params(64, 16, 8, 16, 0.1, select_mode=2, chunk=49), kara.EINVAL),
    ]
    for c, pp, want in cases:
        st = kara._lib.kara_compress_batch(ctypes.byref(c), ctypes.byref(pp), ctypes.byref(b), ws, 4, ws, ws,
                                           None, None, None, ws, 1 << 30, ws, None, None)
        assert st == want, (c.head_dim, pp.W, st)
    # workspace too small is refused before launching
    st = kara._lib.kara_compress_batch(ctypes.byref(fake_cache(kara)), ctypes.byref(p), ctypes.byref(b), ws, 4,
                                       ws, ws, None, None, None, ws, 1, ws, None, None)
    assert st == kara.EWORKSPACE


def test_batch_groups_query(kara, monkeypatch):
    """kara_batch_groups: argument checks as the entry points, one group for a
    single sequence, and the KARA_BATCH_GROUPS override clamped to [1, min(n, 64)]
    (no device is touched on these paths)."""
    p = kara.params(64, 16, 8, 16, 0.1)
    bad = kara._lib.kara_batch_groups(ctypes.byref(fake_cache(kara, head_dim=96)), ctypes.byref(p),
                                      ctypes.byref(kara.Batch(5, 16, 16, 16, 16)))
    assert bad == kara.EUNSUPPORTED
    c = fake_cache(kara)
    assert kara.kara_batch_groups(c, p, kara.Batch(1, 16, 16, 16, 16)) == 1
    for env, n, want in (("3", 5, 3), ("100", 5, 5), ("100", 90, 64), ("0", 5, 1), ("-2", 5, 1)):
        monkeypatch.setenv("KARA_BATCH_GROUPS", env)
        assert kara.kara_batch_groups(c, p, kara.Batch(n, 16, 16, 16, 16)) == want, env


def test_workspace_size_grows_with_batch(kara):
    c = fake_cache(kara)
    p = kara.params(64, 16, 8, 16, 0.1)
    a, b = kara.kara_workspace_size(c, p, 1), kara.kara_workspace_size(c, p, 10)
    assert 0 < a < b
    assert kara.kara_workspace_size(fake_cache(kara, head_dim=96), p, 1) == 0


def test_decode_and_ring_argument_checks(kara):
    """The decode-attention and query-ring entry points refuse bad arguments on
    the host with a status; none of these calls launches anything."""
    L = kara._lib
    ws = ctypes.c_void_p(16)
    c = fake_cache(kara)

    def dec(cache=c, layer=0, n=1, lens=ws, bt=ws, bts=16, q=ws, out=ws, w=ws, wb=1 << 30, err=ws):
        return L.kara_decode_attention(ctypes.byref(cache), layer, n, lens, bt, bts, q, out, w, wb, err, None)

    assert dec(cache=fake_cache(kara, head_dim=96)) == kara.EUNSUPPORTED
    assert dec(cache=fake_cache(kara, k=None)) == kara.EINVAL
    assert dec(layer=-1) == kara.EINVAL and dec(layer=1) == kara.EINVAL    # the fake cache has 1 layer
    assert dec(n=-1) == kara.EINVAL and dec(bts=0) == kara.EINVAL
    assert dec(n=0) == kara.OK                                              # nothing to do
    assert dec(lens=None) == kara.EINVAL and dec(bt=None) == kara.EINVAL and dec(err=None) == kara.EINVAL
    assert dec(q=ctypes.c_void_p(18)) == kara.EINVAL                         # q not 16-byte aligned
    assert dec(n=65536) == kara.EUNSUPPORTED
    assert dec(w=None) == kara.EWORKSPACE and dec(wb=1) == kara.EWORKSPACE
    assert kara.kara_decode_workspace_size(c, 1, 16) > 0

    p = kara.params(64, 16, 8, 16, 0.1)
    b = kara.Batch(1, 16, 16, 16, 16)
    bn = kara.Batch(-1, 16, 16, 16, 16)
    assert L.kara_compact_queries(ctypes.byref(c), ctypes.byref(p), ctypes.byref(bn), ws, ws, None) == kara.EINVAL
    assert L.kara_append_queries(ctypes.byref(c), ctypes.byref(p), ctypes.byref(bn), ws, None) == kara.EINVAL
    b0 = kara.Batch(0, 16, 16, 16, 16)
    assert L.kara_compact_queries(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b0), ws, ws, None) == kara.OK
    assert L.kara_append_queries(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b0), ws, None) == kara.OK
    assert L.kara_compact_queries(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b), None, ws, None) == kara.EINVAL
    assert L.kara_append_queries(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b), None, None) == kara.EINVAL
    assert L.kara_append_queries(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b), ctypes.c_void_p(24),
                                 None) == kara.EINVAL                      # q_new not 16-byte aligned
    bad = kara.params(64, 16, 8, 0, 0.1)
    assert L.kara_compact_queries(ctypes.byref(c), ctypes.byref(bad), ctypes.byref(b), ws, ws, None) == kara.EINVAL
