"""Benchmark of the Kara compression step on GB300: one JSON line on stdout.

A step is one kara_compress_batch over a whole batch (plan, score, select,
compact, commit) on inputs already resident in HBM.  Default workload: the
Qwen3-14B-shaped batch (128 sequences x 40 layers x 8 KV heads = 40960
windows, W 1024).  `--impl reference` times the CPU oracle on the host cores
on a bounded sample of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kara|reference]
                       [--config qwen3_14b|qwen3_4b|llama_8b|tiny]
Multi-GPU: launched by torch.distributed.run, each rank compresses its own
batch (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "compressed windows/sec (seq·layer·kv-head), HBM GB/s, % of roofline"
# ex2 results per clock per SM that the special-function pipe can deliver: the
# scoring kernel's ncu capture executes 13.2 ex2 per clock per SM with that pipe
# at 42.4 % of its peak instruction rate, which puts the peak near 32.
EXP_PER_CLK_SM = 32


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def exp_diagnostic(spec, nwin, causal, score_ms, mhz, n_sm):
    """The exponential unit as a third bound of the scorer, reported beside the
    contract's two: one exponential per (head, query, key) of every window (the
    causal mask leaves W(W+1)/2 pairs per head), the time they take at the
    pipe's peak rate on n_sm SMs at mhz, and the rate the scorer reached."""
    pairs = spec.W * (spec.W + 1) // 2 if causal else spec.W * spec.W
    count = nwin * spec.G * pairs
    out = {"count": count, "peak_per_clk_per_sm": EXP_PER_CLK_SM, "sms": n_sm, "t_ms": None,
           "achieved_per_clk_per_sm": None}
    if mhz:
        hz = n_sm * mhz * 1e6
        out["t_ms"] = count / (EXP_PER_CLK_SM * hz) * 1e3
        out["achieved_per_clk_per_sm"] = count / (score_ms * 1e-3) / hz
    return out


def traffic_record(name):
    """A committed ncu traffic record under profiles/, or None when the sources
    it was taken from have changed since the capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", name)) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        return rec if h.hexdigest()[:16] == rec["sources_sha256_16"] else None
    except Exception:
        return None


def measured_traffic(nwin):
    """DRAM bytes of one scoring launch from the committed ncu capture, scaled by
    windows; None when the scorer's sources changed since the capture."""
    rec = traffic_record("score_sp_traffic.json")
    return rec["bytes_per_window"] * nwin if rec else None


def measured_decode_traffic(kv_bytes):
    """DRAM bytes of one decode split launch from the committed ncu capture,
    scaled by the launch's K/V bytes; None when the sources changed since."""
    rec = traffic_record("decode_split_traffic.json")
    return round(rec["dram_bytes"] / rec["kv_bytes_captured"] * kv_bytes) if rec else None


def algorithmic(spec, lengths):
    """Per-step algorithmic work: QK^T FLOPs of the scoring and minimum bytes.

    FLOPs/window = 2*G*W^2*D.  Bytes/window = Q window (G*W*D*2) + K window
    (W*D*2) read once + V rows read and K/V rows written for the o + R + B rows
    each window keeps (o = (L - W) mod 16)."""
    G, W, D = spec.hq // spec.hkv, spec.W, spec.d
    per_layer_head = spec.layers * spec.hkv
    flops = 2.0 * G * W * W * D * spec.n_seq * per_layer_head
    score_bytes = (G * W * D * 2 + W * D * 2) * spec.n_seq * per_layer_head
    rows = sum(((int(L) - W) % spec.block) + spec.R + spec.B for L in lengths)
    compact_bytes = rows * per_layer_head * D * 2 * 3     # V read, K and V written (K read: in score_bytes)
    return flops, score_bytes, compact_bytes


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        try:
            rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        except Exception:
            return out
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, reasons = [], set()
        mx = None
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except (ValueError, IndexError):
                continue
            for nm, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if sm:
            out.update(sm_mhz=statistics.median(sm), sm_max_mhz=mx, reasons=sorted(reasons), samples=len(sm))
        return out


def cpu_oracle_sample(wl_dev, seqs, layers_sample, threads=None, keep=False):
    """Time the oracle (as it stands) on a bounded sample: the windows of a few
    sequences and layers of the same workload, on `threads` host threads (all
    cores by default).  Returns (windows/s, seconds, threads, windows), and with
    keep=True also what the parity check needs: the oracle's scores, cand and
    kept, the shape and the host sub-workload."""
    import oracle
    sub = synth.host_subset(wl_dev, seqs)
    spec = sub.spec.with_(layers=layers_sample)
    q = sub.q[:, :layers_sample].contiguous()
    k = sub.k[:layers_sample].contiguous()
    v = sub.v[:layers_sample].contiguous()
    sh = oracle.make_shape(spec.n_seq, spec.layers, spec.hq, spec.hkv, spec.d, spec.block, spec.W, spec.B,
                           spec.K, spec.R, spec.lam, sub.bt_stride, sub.num_blocks)
    threads = threads or oracle.max_threads()
    t0 = time.perf_counter()
    sc = oracle.scores(sh, q, k, sub.block_table, sub.lengths, nthreads=threads)
    cand, kept = oracle.select_batch(sc, spec.K, spec.R, spec.lam, nthreads=threads)
    st = oracle.compact(sh, k, v, sub.block_table, sub.lengths, kept, sub.fresh)[0]
    dt = time.perf_counter() - t0
    assert st == oracle.OK
    nwin = spec.n_seq * spec.layers * spec.hkv
    if keep:
        return nwin / dt, dt, threads, nwin, dict(sc=sc, cand=cand, kept=kept, sh=sh, sub=sub, k=k, v=v)
    return nwin / dt, dt, threads, nwin


def window_rows(kpool, vpool, bt, lengths, W, B, R, bs, layers):
    """K and V rows of the rebuilt region [p0*bs, L') of each sequence's window,
    read through a table: [seq] -> (k [rows][layers][hkv][D], v alike), raw bits."""
    out = []
    for s in range(bt.shape[0]):
        L = int(lengths[s])
        p0 = (L - W) // bs
        x = np.arange(p0 * bs, L - (W - B) + R)
        blk = np.asarray(bt[s])[x // bs].astype(np.int64)
        slot = x % bs
        if isinstance(kpool, torch.Tensor):      # gathered on the device, then copied
            bi = torch.from_numpy(blk).to(kpool.device)
            si = torch.from_numpy(slot).to(kpool.device)
            out.append((kpool[:layers][:, bi, :, si, :].cpu().numpy(),
                        vpool[:layers][:, bi, :, si, :].cpu().numpy()))
        else:
            out.append((kpool[:layers][:, blk, :, slot, :], vpool[:layers][:, blk, :, slot, :]))
    return out


def parity_sample(kara, spec, c, p, b, bt, bt0, fresh, freed, new_len, ws, err, wl, seqs, layers, ref):
    """The GPU's outputs on the oracle's sample windows, compared with the oracle:
    scores (max relative error), selection (exact kept/cand rows: on the oracle's
    own scores, on the windows whose oracle selection is stable under 1e-4
    relative noise, and on the GPU's scores, where it must be exact), and
    compaction (the bytes of every rebuilt row, the oracle compacting with the
    GPU's kept)."""
    import oracle
    dev = wl.q.device
    scores = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.C, dtype=torch.float32, device=dev)
    cand = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.K, dtype=torch.int32, device=dev)
    kept = torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.R, dtype=torch.int32, device=dev)
    bt.copy_(bt0)
    kara.kara_compress_batch(c, p, b, fresh, freed, new_len, ws, err, scores_out=scores, cand_out=cand,
                             kept_out=kept)
    assert kara.kara_get_error(err) == 0
    g_sc = scores[seqs, :layers].cpu().numpy()
    g_cand = cand[seqs, :layers].cpu().numpy()
    g_kept = kept[seqs, :layers].cpu().numpy()
    g_bt = bt[seqs].cpu().numpy()
    g_rows = window_rows(wl.k.view(torch.int16), wl.v.view(torch.int16), g_bt, wl.lengths[seqs].cpu().numpy(),
                         spec.W, spec.B, spec.R, spec.block, layers)
    bt.copy_(bt0)
    torch.cuda.synchronize()
    rel = np.abs(g_sc.astype(np.float64) - ref["sc"].astype(np.float64)) / np.maximum(np.abs(ref["sc"]), 1e-30)
    C = spec.C
    flat = ref["sc"].reshape(-1, C)
    base = ref["kept"].reshape(-1, spec.R)
    rng = np.random.default_rng(0)
    stable = np.ones(flat.shape[0], bool)
    for _ in range(6):
        pert = (flat * (1 + 1e-4 * rng.uniform(-1, 1, flat.shape))).astype(np.float32)
        stable &= np.all(oracle.select_batch(pert, spec.K, spec.R, spec.lam)[1] == base, axis=-1)
    kept_eq = np.all(g_kept.reshape(-1, spec.R) == base, axis=-1)
    cand_eq = np.all(g_cand.reshape(-1, spec.K) == ref["cand"].reshape(-1, spec.K), axis=-1)
    o_cand, o_kept = oracle.select_batch(g_sc.reshape(-1, C), spec.K, spec.R, spec.lam)
    same_in = np.all(o_kept == g_kept.reshape(-1, spec.R), axis=-1) & np.all(o_cand == g_cand.reshape(-1, spec.K),
                                                                              axis=-1)
    sub = ref["sub"]
    st, k2, v2, bt2, _, nl2 = oracle.compact(ref["sh"], ref["k"], ref["v"], sub.block_table, sub.lengths, g_kept,
                                             sub.fresh)
    assert st == oracle.OK
    o_rows = window_rows(k2, v2, bt2, sub.lengths.numpy(), spec.W, spec.B, spec.R, spec.block, layers)
    mism = sum(int(np.count_nonzero(a.view(np.uint16) != b.view(np.uint16)))
               for (ga, gb), (oa, ob) in zip(g_rows, o_rows) for a, b in ((ga, oa), (gb, ob)))
    nbytes = sum(a.size * 2 for ga, gb in g_rows for a in (ga, gb))
    n = flat.shape[0]
    return {"sample": f"{n} windows ({len(seqs)} sequences x {layers} layers x {spec.hkv} KV heads) of the "
                      f"timed workload; oracle: fp64 scores, selection, compaction",
            "max_rel_score_err": float(rel.max()), "score_rtol": 1e-3,
            "kept_exact": float(kept_eq.mean()), "cand_exact": float(cand_eq.mean()),
            "stable_windows": int(stable.sum()), "kept_exact_on_stable": float(kept_eq[stable].mean())
            if stable.any() else None,
            "selection_exact_given_gpu_scores": float(same_in.mean()),
            "compaction_bytes_compared": int(nbytes), "compaction_byte_mismatches": mism}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            # each rank's GPU is bound before NCCL sets up its communicator
            torch.cuda.set_device(local)
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sample_layers(wl, seqs, target_s=12.0, threads=None):
    """Layers of the oracle sample: enough for about target_s seconds of host
    work (timed from a one-layer probe), at most the workload's layer count."""
    _, dt, _, _ = cpu_oracle_sample(wl, seqs, 1, threads=threads)
    return max(1, min(wl.spec.layers, int(round(target_s / max(dt, 1e-3)))))


def run_reference(args, ws, rank):
    """The oracle arm: each step is a bounded sample of the workload on the host cores."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    spec = synth.SPECS[args.config]
    seqs = list(range(min(2, spec.n_seq)))
    wl = synth.generate(spec.with_(n_seq=len(seqs)), device="cpu")
    # only this rank works, so it takes every host core it may run on (under
    # torchrun each process starts with OMP_NUM_THREADS=1)
    thr = len(os.sched_getaffinity(0))
    layers_sample = sample_layers(wl, seqs, threads=thr)
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, seqs, layers_sample, threads=thr)
    times = []
    nwin = 0
    for _ in range(args.steps):
        rate, dt, thr, nwin = cpu_oracle_sample(wl, seqs, layers_sample, threads=thr)
        times.append(dt)
    t = statistics.median(times)
    val = nwin / t
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "windows/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.config}: oracle sample of {nwin} windows "
                                   f"({len(seqs)} sequences x {layers_sample} layers x {spec.hkv} KV heads)"},
            "cpu_baseline": {"value": val, "unit": "windows/s", "cores": thr, "kind": "oracle",
                             "sample": f"{nwin} windows of the {args.config} workload per step"},
            "e2e": {"value": val, "unit": "windows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


VARIANT_CODES = {"bidirectional": 0, "causal": 1, "token2chunk": 0, "top_r": 1, "fixed_chunk": 2}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kara", choices=["kara", "reference"])
    ap.add_argument("--config", default="qwen3_14b", choices=sorted(synth.SPECS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--n-seq", type=int, default=None, help="override the workload's sequence count")
    ap.add_argument("--score-mode", default="bidirectional", choices=["bidirectional", "causal"],
                    help="scoring variant (causal is the ablation without bidirectional attention)")
    ap.add_argument("--select-mode", default="token2chunk", choices=["token2chunk", "top_r", "fixed_chunk"],
                    help="selection variant (top_r and fixed_chunk are the ablations of Token2Chunk)")
    ap.add_argument("--chunk", type=int, default=0, help="chunk length for --select-mode fixed_chunk")
    ap.add_argument("--q-ring", action="store_true",
                    help="treat the window queries as a ring and add kara_compact_queries to every step")
    ap.add_argument("--layers", type=int, default=None, help="override the workload's layer count")
    ap.add_argument("--profile-kernel", choices=["score", "select", "compact"], default=None,
                    help="only run one entry point `--steps` times (for ncu captures); prints no JSON")
    ap.add_argument("--sweep", action="store_true",
                    help="periodic-policy sweep on the Qwen3-4B shape: one JSON line per compression event")
    ap.add_argument("--serve-sim", action="store_true",
                    help="admission scheduler over a fixed block pool, with and without periodic compression")
    ap.add_argument("--decode", action="store_true",
                    help="decode attention over the paged cache (one layer of the workload): one JSON line")
    ap.add_argument("--sweep-batches", default="1,8,32,128,256")
    ap.add_argument("--sweep-windows", default="128,256,512,1024,2048")
    args = ap.parse_args()
    ws_, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws_, rank)
        return

    from decode_kv_cache_03_gb300 import build as kbuild
    if rank == 0 or ws_ == 1:
        kbuild.build()
    barrier(ws_)
    from decode_kv_cache_03_gb300 import kara

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.sweep:
        run_sweep(args, dev)
        return
    if args.decode:
        run_decode(args, dev, kara)
        return
    if args.serve_sim:
        run_serve_sim(args, dev)
        return
    spec = synth.SPECS[args.config].with_(seed=synth.SPECS[args.config].seed + 97 * rank)
    if args.n_seq:
        spec = spec.with_(n_seq=args.n_seq)
    if args.layers:
        spec = spec.with_(layers=args.layers)
    wl = synth.generate(spec, device=dev)
    torch.cuda.synchronize()
    c = kara.cache(wl.k, wl.v, spec.hq)
    p = kara.params(spec.W, spec.B, spec.K, spec.R, spec.lam, VARIANT_CODES[args.score_mode],
                    VARIANT_CODES[args.select_mode], args.chunk)
    lengths_h = wl.lengths.cpu()
    nn, no, tn, to = kara.kara_plan(p, spec.block, lengths_h, wl.bt_stride)
    bt0 = wl.block_table.clone()
    bt = wl.block_table
    b = kara.batch(wl.lengths, bt, wl.q)
    fresh = wl.fresh
    freed = torch.empty(to, dtype=torch.int32, device=dev)
    new_len = torch.empty(spec.n_seq, dtype=torch.int32, device=dev)
    ws = torch.empty(kara.kara_workspace_size(c, p, spec.n_seq), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for row in ev:                         # torch creates the CUDA event on its first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    # --q-ring: the window queries are a ring (row = position mod W) that each step
    # compacts with K/V; kept goes to a caller buffer for kara_compact_queries
    kept_buf = (torch.empty(spec.n_seq, spec.layers, spec.hkv, spec.R, dtype=torch.int32, device=dev)
                if args.q_ring else None)

    if args.profile_kernel:
        profile_kernel(args, kara, spec, wl, c, p, b, fresh, freed, new_len, ws, err)
        return
    groups = kara.kara_batch_groups(c, p, b)

    def step(events=None):
        bt.copy_(bt0)                      # every step compresses the same trailing windows
        kara.kara_compress_batch(c, p, b, fresh, freed, new_len, ws, err, kept_out=kept_buf, stream=stream,
                                 phase_events=events[:5] if events else None)
        if args.q_ring:
            kara.kara_compact_queries(c, p, b, kept_buf, err, stream)
            if events:
                events[5].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = kara.kara_get_error(err)
    if status != 0:
        raise SystemExit(f"compression reported {kara.status_string(status)}")

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(ws_)
        torch.cuda.synchronize()
        t0.record(stream)
        for i in range(args.steps):
            step(ev[i])
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(ws_)
    total_ms = max_over_ranks(t0.elapsed_time(t1), ws_)
    ms = total_ms / args.steps
    # phases: scoring (every group's); then what the selection, checks, copy and
    # commit add after it (in groups, most of it ran under the next group's scoring)
    score_ms = statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps))
    after_ms = statistics.mean(ev[i][2].elapsed_time(ev[i][4]) for i in range(args.steps))
    qring_ms = statistics.mean(ev[i][4].elapsed_time(ev[i][5]) for i in range(args.steps)) if args.q_ring else None
    status = kara.kara_get_error(err)
    if status != 0:
        raise SystemExit(f"compression reported {kara.status_string(status)}")

    # end to end through the public API with host buffers: the scheduler's tables,
    # lengths and fresh ids go up from pinned memory, the new tables, lengths,
    # freed ids and status come back, every step
    h_len = lengths_h.pin_memory()
    h_bt = bt0.cpu().pin_memory()
    h_fresh = fresh.cpu().pin_memory()
    h_bt_out = torch.empty_like(h_bt).pin_memory()
    h_len_out = torch.empty_like(h_len).pin_memory()
    h_freed = torch.empty(to, dtype=torch.int32).pin_memory()
    h_err = torch.empty(1, dtype=torch.int32).pin_memory()
    d_len = torch.empty_like(wl.lengths)
    d_fresh = torch.empty_like(fresh)
    b_e2e = kara.batch(d_len, bt, wl.q)
    e2e_steps = args.e2e_steps or args.steps
    e2e_ms = []
    for i in range(e2e_steps + 1):
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        d_len.copy_(h_len, non_blocking=True)
        bt.copy_(h_bt, non_blocking=True)
        d_fresh.copy_(h_fresh, non_blocking=True)
        kara.kara_compress_batch(c, p, b_e2e, d_fresh, freed, new_len, ws, err, kept_out=kept_buf, stream=stream)
        if args.q_ring:
            kara.kara_compact_queries(c, p, b_e2e, kept_buf, err, stream)
        h_bt_out.copy_(bt, non_blocking=True)
        h_len_out.copy_(new_len, non_blocking=True)
        h_freed.copy_(freed, non_blocking=True)
        h_err.copy_(err, non_blocking=True)
        a1.record(stream)
        a1.synchronize()
        if i > 0:
            e2e_ms.append(a0.elapsed_time(a1))
    assert int(h_err[0]) == 0
    e2e_ms_v = max_over_ranks(statistics.mean(e2e_ms), ws_)
    select_ms, compact_ms = standalone_phases(kara, spec, c, p, b, bt, bt0, fresh, freed, new_len, ws, err, stream)
    h2d = (h_len.numel() + h_bt.numel() + h_fresh.numel()) * 4
    d2h = (h_bt_out.numel() + h_len_out.numel() + h_freed.numel() + 1) * 4

    nwin = spec.n_windows
    flops, score_bytes, compact_bytes = algorithmic(spec, lengths_h.tolist())
    hbm, tf_burst, tf_sus, src = peaks()
    achieved_tflops = flops / (score_ms * 1e-3) / 1e12
    value = nwin * ws_ / (ms * 1e-3)
    clocks = clk.summary()
    # the scorer's bound is the slower of its QK^T FLOPs at the sustained bf16 peak
    # and its algorithmic bytes (Q and K windows) at the measured HBM copy rate
    if score_bytes / (hbm * 1e9) > flops / (tf_sus * 1e12):
        ach = score_bytes / (score_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_kind": f"{src} HBM copy"}
    else:
        roof = {"bound": "tensor", "achieved": achieved_tflops, "peak": tf_sus, "unit": "TFLOP/s",
                "frac": achieved_tflops / tf_sus, "peak_kind": f"{src} sustained bf16",
                "frac_vs_burst": achieved_tflops / tf_burst}
    roof.update({"traffic": measured_traffic(nwin) if (args.config == "qwen3_14b" and args.score_mode == "bidirectional")
                 else None,
                 "traffic_unit": "bytes per launch (DRAM read + write)", "algorithmic_bytes": score_bytes,
                 "kernel": "window scoring (QK^T, softmax, column sums)"})
    line = {
        "metric": METRIC, "value": value, "unit": "windows/s", "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.config}: {spec.n_seq} seq x {spec.layers} layers x {spec.hkv} KV heads "
                               f"= {nwin} windows, W {spec.W} (C {spec.C} + B {spec.B}), G {spec.G}, D {spec.d}, "
                               f"Top-K {spec.K}, R {spec.R}",
                   "variant": {"score": args.score_mode, "select": args.select_mode, "chunk": args.chunk},
                   "l2": "inputs larger than L2 (Q windows and K/V pools are tens of GB per step)",
                   "step": "block table restored by a device copy, then kara_compress_batch"
                           + (f" (pipelined in {groups} groups of sequences)" if groups > 1 else ""),
                   "parallelism": f"dp{ws_} (independent batches per GPU)"},
        "roofline": roof,
        "phases_ms": {"score": score_ms, "after_score": after_ms, "groups": groups,
                      "score_gbs": score_bytes / (score_ms * 1e-3) / 1e9,
                      "select_alone": select_ms, "compact_alone": compact_ms,
                      "compact_alone_gbs": compact_bytes / (compact_ms * 1e-3) / 1e9},
        "step_roofline": {"t_flop_ms": flops / (tf_burst * 1e12) * 1e3,
                          "t_hbm_ms": (score_bytes + compact_bytes) / (hbm * 1e9) * 1e3,
                          "frac": max(flops / (tf_burst * 1e12), (score_bytes + compact_bytes) / (hbm * 1e9))
                          / (ms * 1e-3),
                          "exp": exp_diagnostic(spec, nwin, args.score_mode == "causal", score_ms,
                                                clocks.get("sm_mhz") or clocks.get("sm_max_mhz"),
                                                torch.cuda.get_device_properties(dev).multi_processor_count)},
        "e2e": {"value": nwin * ws_ / (e2e_ms_v * 1e-3), "unit": "windows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": None,
        "clocks": clocks,
    }
    line["gpu_launches"] = args.steps * (launches_per_step(spec.W, args.score_mode == "causal", groups)
                                         + (1 if args.q_ring else 0))
    if args.q_ring:
        qbytes = nwin * spec.G * (spec.R + spec.B) * spec.d * 2 * 2
        line["phases_ms"]["compact_queries"] = qring_ms
        line["phases_ms"]["compact_queries_gbs"] = qbytes / (qring_ms * 1e-3) / 1e9
        line["config"]["q_ring"] = "window queries kept as a ring and compacted every step"
    if rank == 0 and ws_ == 1 and not args.no_cpu_baseline:
        sample_seqs = list(range(min(2, spec.n_seq)))
        bt.copy_(bt0)
        torch.cuda.synchronize()
        nl = sample_layers(wl, sample_seqs)
        rate, dt, thr, sw, ref = cpu_oracle_sample(wl, sample_seqs, nl, keep=True)
        line["cpu_baseline"] = {"value": rate, "unit": "windows/s", "cores": thr, "kind": "oracle",
                                "sample": f"{sw} windows ({len(sample_seqs)} sequences x {nl} layers x "
                                          f"{spec.hkv} KV heads) of the same workload, {dt:.1f} s"}
        # the same oracle on one core, over the windows of one sequence and one layer
        rate1, dt1, _, sw1 = cpu_oracle_sample(wl, sample_seqs[:1], 1, threads=1)
        line["cpu_baseline"]["single_core"] = {"value": rate1, "unit": "windows/s", "cores": 1,
                                               "sample": f"{sw1} windows (1 sequence x 1 layer x {spec.hkv} KV "
                                                         f"heads), {dt1:.1f} s"}
        if not args.q_ring and args.score_mode == "bidirectional" and args.select_mode == "token2chunk":
            line["parity"] = parity_sample(kara, spec, c, p, b, bt, bt0, fresh, freed, new_len, ws, err, wl,
                                           sample_seqs, nl, ref)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_ > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_sweep(args, dev):
    """Periodic policy on the Qwen3-4B shape: 512 decode steps per point; every
    128 steps a seeded half of the sequences compresses its trailing window.
    Each event reports the kara_compress_batch time (plan, scoring, selection,
    compaction and table rewrite, CUDA events around the call) and the blocks
    it released.  Points whose memory would exceed `cap` are reported skipped."""
    import math
    from decode_kv_cache_03_gb300 import Compressor
    from decode_kv_cache_03_gb300.periodic import BlockPool, PeriodicSchedule, append_tokens, compress_selected
    hbm, tf_burst, _, src = peaks()
    cap = 0.8 * torch.cuda.get_device_properties(dev).total_memory
    index = 0
    for b in [int(x) for x in args.sweep_batches.split(",")]:
        for W in [int(x) for x in args.sweep_windows.split(",")]:
            spec = synth.sweep_spec(b, W, index)
            index += 1
            block_bytes = spec.layers * spec.hkv * spec.block * spec.d * 2 * 2
            per_new = math.ceil((spec.block - 1 + spec.R + spec.B) / spec.block)
            fresh_per_seq = per_new + 512 // spec.block + 4
            m_max = math.ceil(b / 2)
            need = (16 + b * (W // spec.block + 1 + fresh_per_seq)) * block_bytes \
                + m_max * spec.layers * spec.hq * W * spec.d * 2
            point = {"batch": b, "W": W, "B": spec.B, "K": spec.K, "R": spec.R}
            if need > cap:
                print(json.dumps({"sweep": dict(point, skipped=f"capacity: needs {need / 1e9:.0f} GB")}), flush=True)
                continue
            wl = synth.generate(spec, device=dev, with_q=False, alias_prefix=True, fresh_per_seq=fresh_per_seq)
            gen = torch.Generator(device=dev).manual_seed(1000 + index)
            q = torch.empty(m_max, spec.layers, spec.hq, W, spec.d, dtype=torch.bfloat16, device=dev)
            for i in range(m_max):
                q[i].copy_(torch.randn(spec.layers, spec.hq, W, spec.d, generator=gen, device=dev))
            comp = Compressor(wl.k, wl.v, spec.hq, W, spec.B, spec.K, spec.R, spec.lam)
            lengths = wl.lengths.cpu().tolist()
            stride = wl.bt_stride + 512 // spec.block + 1
            table = torch.full((b, stride), -1, dtype=torch.int32)
            table[:, :wl.bt_stride] = wl.block_table.cpu()
            pool = BlockPool(wl.fresh.cpu().tolist(), pinned=range(wl.prefix_pool))
            sched = PeriodicSchedule(128, 0.5, W, seed=index)
            event = 0
            for step in range(1, 513):
                before = list(lengths)
                append_tokens(lengths, table, pool, spec.block)
                blk = torch.tensor([int(table[s, before[s] // spec.block]) for s in range(b)], device=dev)
                slot = torch.tensor([before[s] % spec.block for s in range(b)], device=dev)
                wl.k[:, blk, :, slot] = torch.randn(b, spec.layers, spec.hkv, spec.d, generator=gen,
                                                    device=dev).to(torch.bfloat16)
                wl.v[:, blk, :, slot] = torch.randn(b, spec.layers, spec.hkv, spec.d, generator=gen,
                                                    device=dev).to(torch.bfloat16)
                if not sched.due(step):
                    continue
                seqs = sched.choose(lengths)
                event += 1
                if not seqs:
                    continue
                m = len(seqs)
                sel_lengths = [lengths[s] for s in seqs]
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                freed, status = compress_selected(comp, seqs, lengths, table, q[:m], pool, events=ev)
                torch.cuda.synchronize()
                ms = ev[0].elapsed_time(ev[1])
                sp = spec.with_(n_seq=m)
                flops, sb, cb = algorithmic(sp, sel_lengths)
                t_roof = max(flops / (tf_burst * 1e12), (sb + cb) / (hbm * 1e9))
                nwin = m * spec.layers * spec.hkv
                print(json.dumps({"sweep": dict(point, event=event, step=step, sequences=m, windows=nwin,
                                                status=status, ms=ms, windows_per_s=nwin / (ms * 1e-3),
                                                freed_blocks=len(freed), roofline_ms=t_roof * 1e3,
                                                roofline_frac=t_roof / (ms * 1e-3), peaks=src)}), flush=True)
            del wl, q, comp
            torch.cuda.empty_cache()


def run_decode(args, dev, kara):
    """Decode attention of one query per (sequence, query head) over one layer of
    the workload's paged cache, every block stored once (no aliased prefix), so
    the K/V bytes really come from HBM.  Bound: HBM; bytes per launch =
    sum_s L_s * Hkv * D * 2 (K and V) * 2 B, plus queries and outputs."""
    spec = synth.SPECS[args.config].with_(layers=1)
    if args.n_seq:
        spec = spec.with_(n_seq=args.n_seq)
    wl = synth.generate(spec, device=dev, alias_prefix=False, with_q=False)
    q = synth.decode_queries(spec, 0, device=dev)
    c = kara.cache(wl.k, wl.v, spec.hq)
    n, bt_stride = wl.block_table.shape
    ws = torch.empty(kara.kara_decode_workspace_size(c, n, bt_stride), dtype=torch.uint8, device=dev)
    out = torch.empty(n, spec.hq, spec.d, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        kara.kara_decode_attention(c, 0, wl.lengths, wl.block_table, q, out, ws, err)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index or 0) as clk:
        e0.record()
        for _ in range(args.steps):
            kara.kara_decode_attention(c, 0, wl.lengths, wl.block_table, q, out, ws, err)
        e1.record()
        torch.cuda.synchronize()
    status = kara.kara_get_error(err)
    if status != 0:
        raise SystemExit(f"decode attention reported {kara.status_string(status)}")
    ms = e0.elapsed_time(e1) / args.steps
    kv_bytes = int(wl.lengths.to(torch.int64).sum()) * spec.hkv * spec.d * 2 * 2
    io_bytes = q.numel() * 2 + out.numel() * 4 + wl.block_table.numel() * 4
    gbs = (kv_bytes + io_bytes) / (ms * 1e-3) / 1e9
    pk = peaks()[0]
    line = {"metric": "decode attention over the paged cache (HBM GB/s)", "value": gbs, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": "bf16 in, f32 accumulation", "data": "synthetic",
            "config": {"workload": f"{args.config}, one layer: {n} sequences x {spec.hq} query / {spec.hkv} KV heads, "
                                   f"D {spec.d}, lengths {spec.len_lo}..{spec.len_hi}, {kv_bytes / 1e9:.2f} GB of K/V",
                       "l2": "K/V larger than L2, every block distinct"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk, "unit": "GB/s", "frac": gbs / pk,
                         "traffic": measured_decode_traffic(kv_bytes),
                         "traffic_unit": "bytes per launch of the split kernel (DRAM read + write)",
                         "algorithmic_bytes": kv_bytes + io_bytes},
            "gpu_launches": 2 * args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_serve_sim(args, dev):
    """The concurrency argument of the pages (summary, "Problem Statement" item 1
    and section 3) on synthetic decoding: requests share a fixed pool of KV
    blocks under the admission scheduler, once without compression and once
    with the periodic policy compressing through kara_compress_batch.  Prints
    one JSON line per run: mean running sequences, tokens decoded, requests
    finished and the device time of the compression calls."""
    from decode_kv_cache_03_gb300 import Compressor
    from decode_kv_cache_03_gb300.periodic import AdmissionScheduler, BlockPool, PeriodicSchedule
    base = synth.sweep_spec(1, 512)
    layers, total, steps, nreq = 4, 16384, 3000, 256
    k = torch.empty(layers, total, base.hkv, base.block, base.d, dtype=torch.bfloat16, device=dev)
    gen = torch.Generator(device=dev).manual_seed(1)
    for l in range(layers):
        k[l] = torch.randn(total, base.hkv, base.block, base.d, generator=gen, device=dev).to(torch.bfloat16)
    v = torch.randn_like(k)
    rng = torch.Generator().manual_seed(2)
    reqs = [(int(torch.randint(512, 1025, (1,), generator=rng)), int(torch.randint(2048, 6145, (1,), generator=rng)))
            for _ in range(nreq)]

    def q_window(n):
        return torch.randn(n, layers, base.hq, base.W, base.d, generator=gen, device=dev).to(torch.bfloat16)

    for compress in (False, True):
        comp = Compressor(k, v, base.hq, base.W, base.B, base.K, base.R, base.lam)
        sched = AdmissionScheduler(BlockPool(range(total)), reqs, base.block, bt_stride=(1024 + 6144) // 16 + 1)
        schedule = PeriodicSchedule(128, 0.5, base.W, seed=3)
        running, ev_ms, freed = [], [], 0
        t0 = time.perf_counter()
        for step in range(1, steps + 1):
            sched.admit()
            sched.step()
            running.append(len(sched.running))
            if compress and schedule.due(step):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                freed += sched.compress(comp, schedule, q_window)
                e1.record()
                torch.cuda.synchronize()
                ev_ms.append(e0.elapsed_time(e1))
        wall = time.perf_counter() - t0
        line = {"metric": "serving simulation: tokens decoded in a fixed block pool", "value": sched.tokens,
                "unit": "tokens", "steps": steps, "compression": compress,
                "mean_running": statistics.mean(running), "max_running": max(running),
                "finished": len(sched.finished), "compress_events": len(ev_ms), "blocks_freed": freed,
                "compress_ms_mean": statistics.mean(ev_ms) if ev_ms else 0.0, "host_seconds": wall,
                "config": {"pool_blocks": total, "block": base.block, "layers": layers,
                           "heads": f"{base.hq}/{base.hkv}", "D": base.d, "W": base.W, "B": base.B, "K": base.K,
                           "R": base.R, "requests": nreq, "prompt": "512..1024", "generate": "2048..6144",
                           "policy": "every 128 steps, half of the eligible sequences"},
                "data": "synthetic"}
        print(json.dumps(line), flush=True)


def standalone_phases(kara, spec, c, p, b, bt, bt0, fresh, freed, new_len, ws, err, stream, reps=3):
    """Selection (kara_select) and checks + compaction + commit (kara_compact)
    timed through their own entry points on the step's data, outside the timed
    step: inside kara_compress_batch they overlap the scoring when it runs in
    groups.  Returns their mean times in ms."""
    dev = bt.device
    scores = torch.empty(spec.n_windows, spec.C, dtype=torch.float32, device=dev)
    cand = torch.empty(spec.n_windows, spec.K, dtype=torch.int32, device=dev)
    kept = torch.empty(spec.n_windows, spec.R, dtype=torch.int32, device=dev)
    bt.copy_(bt0)
    kara.kara_compress_batch(c, p, b, fresh, freed, new_len, ws, err, scores, cand, kept, stream=stream)
    sel, cmp_ = [], []
    for _ in range(reps):
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        bt.copy_(bt0)
        e0.record(stream)
        kara.kara_select(p, spec.n_windows, scores, cand, kept, stream)
        e1.record(stream)
        kara.kara_compact(c, p, b, kept, fresh, freed, new_len, err, ws, stream)
        e2.record(stream)
        e2.synchronize()
        sel.append(e0.elapsed_time(e1))
        cmp_.append(e1.elapsed_time(e2))
    status = kara.kara_get_error(err)
    if status != 0:
        raise SystemExit(f"compaction reported {kara.status_string(status)}")
    bt.copy_(bt0)
    torch.cuda.synchronize()
    return statistics.mean(sel), statistics.mean(cmp_)


def launches_per_step(W, causal, groups=1):
    """Kernels of this library per kara_compress_batch: plan, score, select, the
    fresh-id and kept-row checks, compact, commit.  Scoring is the single-pass
    kernel plus the exact recompute of marked windows (two launches).  In
    groups, each group has its own score, select, kept-check and compact
    launches; plan, fresh-id check and commit run once."""
    score = 2
    return 6 + score if groups <= 1 else 3 + groups * (score + 3)


def profile_kernel(args, kara, spec, wl, c, p, b, fresh, freed, new_len, ws, err):
    """Runs one entry point on the resident workload `--steps` times (ncu target)."""
    nwin = spec.n_windows
    scores = torch.empty(nwin, spec.C, dtype=torch.float32, device=wl.q.device)
    kept = torch.empty(nwin, spec.R, dtype=torch.int32, device=wl.q.device)
    kara.kara_score(c, p, b, scores, ws, err)
    kara.kara_select(p, nwin, scores, None, kept)
    torch.cuda.synchronize()
    bt0 = wl.block_table.clone()
    for _ in range(args.steps):
        if args.profile_kernel == "score":
            kara.kara_score(c, p, b, scores, ws, err)
        elif args.profile_kernel == "select":
            kara.kara_select(p, nwin, scores, None, kept)
        else:
            wl.block_table.copy_(bt0)
            kara.kara_compact(c, p, b, kept, fresh, freed, new_len, err, ws)
    torch.cuda.synchronize()
    status = kara.kara_get_error(err)
    if status != 0:
        raise SystemExit(f"{args.profile_kernel} reported {kara.status_string(status)}")
    print(f"profiled {args.profile_kernel} x{args.steps} on {nwin} windows", flush=True)


if __name__ == "__main__":
    main()
