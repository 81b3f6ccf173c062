"""The bench's reference arm on CPU: the oracle timed on a bounded sample of the
tiny workload, one JSON line with the keys the bench contract names; under two
ranks (as torchrun launches it) rank 0 alone prints and rank 1 exits 0."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CMD = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
       "--steps", "1", "--warmup", "0"]


def _lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_prints_one_contract_line():
    p = subprocess.run(CMD, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = _lines(p.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference"
    assert d["unit"] == "windows/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 0 and d["data"] == "synthetic"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]


@pytest.mark.timeout(600)
def test_reference_arm_under_two_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   LOCAL_RANK=str(rank), WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen(CMD[:1] + CMD[1:] + ["--gpus", "2"], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=600) for p in procs]
    for p, (_, err) in zip(procs, outs):
        assert p.returncode == 0, err[-2000:]
    assert len(_lines(outs[0][0])) == 1 and _lines(outs[0][0])[0]["n_gpus"] == 2
    assert _lines(outs[1][0]) == []


def test_exp_diagnostic_counts():
    """The exponential-unit diagnostic: G*W^2 exponentials per window (W(W+1)/2
    pairs per head under the causal mask) and their time at the peak rate."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    spec = synth.SPECS["qwen3_14b"]
    d = bench.exp_diagnostic(spec, spec.n_windows, False, 64.0, 2000.0, 100)
    assert d["count"] == 40960 * 5 * 1024 * 1024
    hz = 100 * 2000e6
    assert d["t_ms"] == pytest.approx(d["count"] / (bench.EXP_PER_CLK_SM * hz) * 1e3)
    assert d["achieved_per_clk_per_sm"] == pytest.approx(d["count"] / 64e-3 / hz)
    c = bench.exp_diagnostic(spec, 3, True, 1.0, None, 100)
    assert c["count"] == 3 * 5 * (1024 * 1025 // 2) and c["t_ms"] is None
