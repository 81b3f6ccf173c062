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
