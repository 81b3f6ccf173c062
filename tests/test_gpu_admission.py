"""The admission scheduler driving the real library: a run with
kara_compress_batch must follow, step for step, the run with the host
stand-in of the table rule (lengths, tables and free lists identical), and the
block accounting must hold throughout."""
import pytest
import torch

from _cases import random_spec
from _gpu import lib
from test_admission_host import BS, HostCompressor, check_accounting

pytestmark = pytest.mark.gpu


def test_scheduler_with_the_library_matches_the_host_rule():
    lib()
    from decode_kv_cache_03_gb300 import Compressor
    from decode_kv_cache_03_gb300.periodic import AdmissionScheduler, BlockPool, PeriodicSchedule
    total = 700
    spec = random_spec(620, G=2, hkv=2, W=256, B=32, D=128, n_seq=1, layers=2, K=16, R=44)
    # a pool of `total` blocks with random contents
    k = torch.randn(spec.layers, total, spec.hkv, BS, spec.d, device="cuda").to(torch.bfloat16)
    v = torch.randn_like(k)
    comp = Compressor(k, v, spec.hq, spec.W, spec.B, spec.K, spec.R, spec.lam)
    host = HostCompressor(spec.W, spec.B, spec.K, spec.R)
    gen = torch.Generator(device="cuda").manual_seed(3)

    def q_window(n):
        return torch.randn(n, spec.layers, spec.hq, spec.W, spec.d, generator=gen, device="cuda").to(torch.bfloat16)

    rng = torch.Generator().manual_seed(5)
    reqs = [(int(torch.randint(300, 400, (1,), generator=rng)), int(torch.randint(300, 900, (1,), generator=rng)))
            for _ in range(40)]
    a = AdmissionScheduler(BlockPool(range(total)), reqs, BS, bt_stride=96)
    b = AdmissionScheduler(BlockPool(range(total)), reqs, BS, bt_stride=96)
    sa, sb = PeriodicSchedule(64, 0.5, spec.W, seed=7), PeriodicSchedule(64, 0.5, spec.W, seed=7)
    events = 0
    for step in range(1, 901):
        a.admit(), b.admit()
        a.step(), b.step()
        if sa.due(step):
            fa = a.compress(comp, sa, q_window)
            fb = b.compress(host, sb, lambda n: None)
            assert fa == fb
            events += fa > 0
        check_accounting(a, total)
        assert a.running == b.running and a.pool.free == b.pool.free and a.finished == b.finished
    assert events > 3 and a.finished
