"""The compaction's input checks on the GPU, against the oracle's statuses.

A fresh id the plan consumes must be new -- not an earlier consumed id, not a
block any table of the batch still lists -- and a kept row must be strictly
increasing in [0, C).  On a violation the device records the oracle's status
and writes no block at all: the K/V pools, the tables and the lengths are left
byte for byte as they were.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _cases import random_spec
from _gpu import lib, run_compress, to_device

pytestmark = pytest.mark.gpu


def _same_bits(a, b):
    """Byte-for-byte equality (the pools' unwritten slots hold a NaN canary)."""
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _spec():
    return random_spec(17, W=64, B=16, D=64, n_seq=3, layers=2, R=10, len_lo=100, len_hi=180)


def _consumed(wl):
    s = wl.spec
    nn, _ = oracle.plan(wl.lengths, s.W, s.B, s.R, s.block, wl.bt_stride)
    return int(nn.sum())


def _fresh_cases(wl):
    """(name, mutated fresh list) pairs; the oracle gives the expected status."""
    used = _consumed(wl)
    L1 = int(wl.lengths[1])
    out = []
    f = wl.fresh.clone()
    f[used - 1] = f[0]
    out.append(("repeat_in_consumed", f))
    f = wl.fresh.clone()
    f[1] = wl.block_table[2, 0]
    out.append(("prefix_block_of_other_seq", f))
    f = wl.fresh.clone()
    f[0] = wl.block_table[1, (L1 - 1) // wl.spec.block]
    out.append(("old_tail_block_read_by_step", f))
    f = wl.fresh.clone()
    f[used:] = f[0]
    out.append(("repeats_past_consumed_ok", f))
    f = wl.fresh.clone()
    f[2] = wl.num_blocks + 7
    out.append(("outside_pool", f))
    f = wl.fresh.clone()
    f[2] = -3
    f[used - 2] = f[0]
    out.append(("outside_pool_and_repeat", f))
    return out


@pytest.mark.parametrize("idx", range(6))
def test_fresh_ids_checked_before_any_write(idx):
    kara = lib()
    wl = synth.generate(_spec())
    name, fresh = _fresh_cases(wl)[idx]
    wl = synth.Workload(wl.spec, wl.q, wl.k, wl.v, wl.lengths, wl.block_table, fresh, wl.prefix_pool,
                        wl.fresh_base)
    kept = np.tile(np.arange(wl.spec.R, dtype=np.int32), (wl.spec.n_seq, wl.spec.layers, wl.spec.hkv, 1))
    want = oracle.compact(oracle.shape_of(wl), wl.k, wl.v, wl.block_table, wl.lengths, kept, fresh)[0]
    d = to_device(wl)
    k0, v0 = d.k.clone(), d.v.clone()
    out = run_compress(d)
    assert out["status"] == want, name
    if want == oracle.OK:
        assert out["status"] == 0
        return
    assert out["status"] in (kara.EDUPBLOCK, kara.EBADBLOCK)
    assert np.array_equal(out["bt"], wl.block_table.numpy())
    assert np.array_equal(out["new_len"], wl.lengths.numpy())
    assert _same_bits(d.k, k0) and _same_bits(d.v, v0)     # no block written, fresh or live


def _compact_call(kara, d, kept_np, static):
    s = d.spec
    c = kara.cache(d.k, d.v, s.hq)
    p = kara.params(s.W, s.B, s.K, s.R, s.lam)
    bt = d.block_table.clone()
    b = kara.batch(d.lengths, bt, d.q)
    _, _, _, to = kara.kara_plan(p, s.block, d.lengths.cpu(), d.bt_stride)
    freed = torch.full((max(to, 1),), -7, dtype=torch.int32, device="cuda")
    new_len = torch.full((s.n_seq,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kept = torch.from_numpy(kept_np).cuda()
    if static:
        kara.kara_compact_static(c, p, b, kept, d.fresh, freed, new_len, err)
    else:
        ws = torch.empty(kara.kara_workspace_size(c, p, s.n_seq), dtype=torch.uint8, device="cuda")
        kara.kara_compact(c, p, b, kept, d.fresh, freed, new_len, err, ws)
    return kara.kara_get_error(err), bt.cpu().numpy(), new_len.cpu().numpy(), freed.cpu().numpy()


@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("case", ["repeat", "out_of_order", "outside_c", "fresh_is_live"])
def test_compact_entry_points_check_inputs(case, static):
    kara = lib()
    wl = synth.generate(_spec())
    s = wl.spec
    kept = np.tile(np.arange(s.R, dtype=np.int32), (s.n_seq, s.layers, s.hkv, 1))
    fresh = wl.fresh.clone()
    if case == "repeat":
        kept[1, 0, 1, 3] = kept[1, 0, 1, 2]
    elif case == "out_of_order":
        kept[0, 1, 0, 4:6] = kept[0, 1, 0, 4:6][::-1].copy()
    elif case == "outside_c":
        kept[2, 1, 1, -1] = s.C
    else:
        fresh[3] = wl.block_table[0, 1]
    wl = synth.Workload(s, wl.q, wl.k, wl.v, wl.lengths, wl.block_table, fresh, wl.prefix_pool, wl.fresh_base)
    want = oracle.compact(oracle.shape_of(wl), wl.k, wl.v, wl.block_table, wl.lengths, kept, fresh)[0]
    assert want in (oracle.EINVAL, oracle.EDUPBLOCK)
    d = to_device(wl)
    k0, v0 = d.k.clone(), d.v.clone()
    st, bt, new_len, freed = _compact_call(kara, d, kept, static)
    assert st == want
    assert np.array_equal(bt, wl.block_table.numpy())
    assert np.array_equal(new_len, wl.lengths.numpy())
    assert np.all(freed == -7)
    assert _same_bits(d.k, k0) and _same_bits(d.v, v0)


def test_valid_inputs_still_compact_after_a_rejected_call():
    """A rejected call leaves nothing behind: the same context then compacts
    correctly (bit-exact against the oracle)."""
    kara = lib()
    wl = synth.generate(_spec())
    s = wl.spec
    rng = np.random.default_rng(4)
    kept = np.sort(np.stack([rng.choice(s.C, s.R, replace=False) for _ in range(s.n_windows)]), axis=-1)
    kept = kept.astype(np.int32).reshape(s.n_seq, s.layers, s.hkv, s.R)
    d = to_device(wl)
    bad = kept.copy()
    bad[0, 0, 0, :2] = bad[0, 0, 0, 1::-1].copy()
    assert _compact_call(kara, d, bad, False)[0] == kara.EINVAL
    st, bt, new_len, freed = _compact_call(kara, d, kept, False)
    assert st == 0
    st2, k2, v2, bt2, fr2, nl2 = oracle.compact(oracle.shape_of(wl), wl.k, wl.v, wl.block_table, wl.lengths,
                                               kept, wl.fresh)
    assert st2 == oracle.OK
    assert np.array_equal(bt, bt2) and np.array_equal(new_len, nl2) and np.array_equal(freed[:len(fr2)], fr2)
    assert np.array_equal(d.k.view(torch.int16).cpu().numpy().view(np.uint16), k2)
    assert np.array_equal(d.v.view(torch.int16).cpu().numpy().view(np.uint16), v2)
