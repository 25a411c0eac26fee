"""bench.py's command-line contract, on the host (no GPU).

The reference arm (`--impl reference`) times the CPU oracle and prints one
JSON line with the keys the measurement contract names; under torchrun only
rank 0 prints it and every rank exits 0.  The GPU arm refuses to run without
a CUDA device instead of falling back to anything on the CPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--steps", "2", "--warmup", "3", "--workload", "tiny-fbs-sgd"]


def _run(cmd, **kw):
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    env.pop("RANK", None)
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600, **kw)


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check_reference_line(d, n_gpus):
    assert d["impl"] == "reference"
    assert d["unit"] == "IDs/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["n_gpus"] == n_gpus and d["steps"] == 2 and d["warmup"] == 3
    assert d["config"]["workload"] == "tiny-fbs-sgd"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert d["vs_baseline"] is None


def test_reference_arm_prints_one_contract_line():
    r = _run([sys.executable, "bench.py", "--impl", "reference", *ARGS])
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 1)


def test_reference_arm_under_torchrun_prints_from_rank_0_only():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
              "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2",
              "--impl", "reference", *ARGS])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 2)


def test_gpu_arm_refuses_to_run_without_a_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    r = _run([sys.executable, "bench.py", *ARGS])
    assert r.returncode != 0
    assert _json_lines(r.stdout) == []
    assert "CUDA device" in r.stdout + r.stderr
