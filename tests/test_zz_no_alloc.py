"""kara_compact_static, the allocation-free compaction entry point, on the GPU.

Some callers cannot get device memory when compaction runs -- a serving engine
whose pool gave all free HBM to the KV cache, or a host program with no device
allocator -- so they cannot pass a workspace.  kara_compact_static keeps the
per-sequence plan in a fixed array inside the library instead.  These tests
call it through the C ABI and require the same bytes, tables, freed ids,
lengths and status as kara_compact on the same inputs, for two calls in a row
(the second with a smaller batch, so anything the first call left in the shared
array would show up).  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth
from _cases import random_spec
from _gpu import lib, to_device

pytestmark = pytest.mark.gpu


def _inputs(spec, seed):
    wl = synth.generate(spec)
    rng = np.random.default_rng(seed)
    kept = np.sort(np.stack([rng.choice(spec.C, spec.R, replace=False) for _ in range(spec.n_windows)]),
                   axis=-1).astype(np.int32).reshape(spec.n_seq, spec.layers, spec.hkv, spec.R)
    return wl, torch.from_numpy(kept)


def _run(kara, wl, kept, static):
    s = wl.spec
    d = to_device(wl)
    c = kara.cache(d.k, d.v, s.hq)
    p = kara.params(s.W, s.B, s.K, s.R, s.lam)
    bt = d.block_table.clone()
    b = kara.batch(d.lengths, bt, d.q)
    _, _, _, to = kara.kara_plan(p, s.block, wl.lengths, wl.bt_stride)
    freed = torch.full((to,), -9, dtype=torch.int32, device="cuda")
    new_len = torch.full((s.n_seq,), -9, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kept_d = kept.cuda()
    if static:
        kara.kara_compact_static(c, p, b, kept_d, d.fresh, freed, new_len, err)
    else:
        ws = torch.empty(kara.kara_workspace_size(c, p, s.n_seq), dtype=torch.uint8, device="cuda")
        kara.kara_compact(c, p, b, kept_d, d.fresh, freed, new_len, err, ws)
    status = kara.kara_get_error(err)
    return dict(status=status, bt=bt.cpu(), freed=freed.cpu(), new_len=new_len.cpu(),
                k=d.k.view(torch.int16).cpu(), v=d.v.view(torch.int16).cpu())


def test_static_matches_workspace_compaction_on_two_calls_in_a_row():
    kara = lib()
    first = random_spec(91, G=2, hkv=2, W=128, B=16, D=128, n_seq=6, layers=2, R=40, len_lo=128, len_hi=700)
    second = random_spec(92, G=4, hkv=2, W=64, B=16, D=64, n_seq=3, layers=3, R=20, len_lo=64, len_hi=300)
    for spec, seed in ((first, 1), (second, 2)):
        wl, kept = _inputs(spec, seed)
        ref = _run(kara, wl, kept, static=False)
        got = _run(kara, wl, kept, static=True)
        assert ref["status"] == 0 and got["status"] == 0
        for key in ("bt", "freed", "new_len", "k", "v"):
            assert torch.equal(got[key], ref[key]), key


def test_static_reports_device_errors_like_the_workspace_variant():
    kara = lib()
    spec = random_spec(93, G=2, hkv=2, W=64, B=16, D=64, n_seq=3, layers=1, R=16)
    wl, kept = _inputs(spec, 3)
    L = int(wl.lengths[1])
    wl.block_table[1, (L - 1) // 16] = wl.num_blocks + 1
    ref = _run(kara, wl, kept, static=False)
    got = _run(kara, wl, kept, static=True)
    assert ref["status"] == got["status"] == kara.EBADBLOCK
    for key in ("bt", "freed", "new_len", "k", "v"):
        assert torch.equal(got[key], ref[key]), key


def test_static_rejects_batches_above_its_fixed_size():
    kara = lib()
    n = kara.STATIC_MAX_SEQS + 1
    k = torch.zeros(1, 4, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    c = kara.cache(k, k.clone(), 1)
    p = kara.params(64, 16, 8, 16, 0.1)
    lengths = torch.full((n,), 64, dtype=torch.int32, device="cuda")
    bt = torch.zeros(n, 4, dtype=torch.int32, device="cuda")
    q = torch.zeros(n, 1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    b = kara.batch(lengths, bt, q)
    one = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(kara.KaraError) as e:
        kara.kara_compact_static(c, p, b, one, one, one, one, one)
    assert e.value.status == kara.EUNSUPPORTED
