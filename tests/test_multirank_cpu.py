"""The multi-rank path on CPU: two gloo ranks, as bench.py runs them under torchrun.

Each rank compresses its own batch (sequences are independent, so there is no
device collective); the only cross-rank steps are the barrier around the timed
region, the max of the per-rank times and, for a scheduler, the sum of freed
blocks.  This test runs those host-side steps with world size 2 and checks the
aggregates against values computed in the parent process.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_spec(rank):
    base = synth.SPECS["llama_8b"].with_(n_seq=5, layers=1)
    return base.with_(seed=base.seed + 97 * rank)      # the bench's per-rank seeding


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from decode_kv_cache_03_gb300 import kara
    ws, r, local = bench.dist_setup()
    assert (ws, r) == (world, rank)
    spec = _rank_spec(rank)
    wl = synth.generate(spec)
    p = kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam)
    _, _, _, freed = kara.kara_plan(p, spec.block, wl.lengths, wl.bt_stride)
    bench.barrier(ws)
    t_max = bench.max_over_ranks(float(10 + rank), ws)
    tot = torch.tensor([freed], dtype=torch.int64)
    dist.all_reduce(tot)
    out[rank] = (t_max, int(tot.item()), freed)
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_host_side():
    from decode_kv_cache_03_gb300 import build
    build.build()
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=180)
            assert p.exitcode == 0
        res = dict(out)
    expect = []
    from decode_kv_cache_03_gb300 import kara
    for r in range(world):
        spec = _rank_spec(r)
        wl = synth.generate(spec)
        _, _, _, freed = kara.kara_plan(kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam), spec.block,
                                        wl.lengths, wl.bt_stride)
        expect.append(freed)
    for r in range(world):
        t_max, tot, freed = res[r]
        assert t_max == 10.0 + world - 1
        assert freed == expect[r]
        assert tot == sum(expect)
    # ranks work on different batches
    a, b = synth.generate(_rank_spec(0)), synth.generate(_rank_spec(1))
    assert not torch.equal(a.lengths, b.lengths)


def test_reference_arm_under_torchrun_two_ranks():
    """bench.py --impl reference launched as the benchmark driver launches N = 2
    (torchrun, one process per rank, gloo here): rank 0 alone runs the oracle
    on every host core and prints one JSON line; both ranks exit 0."""
    import json
    import subprocess
    import sys
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["cores"] == len(os.sched_getaffinity(0))
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}

