"""The benchmark's reference arm (``bench.py --impl reference``: the fp64
oracle timed on the host cores) needs no GPU, so its JSON contract is
checked here: one line with the arm's own metric, unit and direction, a
cpu_baseline and an e2e that describe this run (no host-device bytes), and
under torchrun with two ranks exactly one line from rank 0 while the other
rank exits 0 without work."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ENV = dict(os.environ, MASTER_ADDR="127.0.0.1", OMP_NUM_THREADS="4")


def _run(args, timeout=300):
    r = subprocess.run(args, cwd=ROOT, env=ENV, capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return lines


def _check_line(d, workload, unit, steps, warmup, n_gpus):
    assert d["impl"] == "reference"
    assert d["unit"] == unit and d["higher_is_better"] is True
    assert d["steps"] == steps and d["warmup"] == warmup and d["n_gpus"] == n_gpus
    assert d["vs_baseline"] is None and d["dtype"] == "f64" and d["scaling"] == "weak"
    assert d["config"]["workload"] == workload
    assert d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == unit
    assert cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == unit
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_decode_line():
    lines = _run([sys.executable, "bench.py", "--impl", "reference", "--workload", "decode_b2_cap256",
                  "--steps", "2", "--warmup", "3"])
    assert len(lines) == 1
    _check_line(json.loads(lines[0]), "decode_b2_cap256", "GB/s", 2, 3, 1)


def test_reference_arm_context_line():
    lines = _run([sys.executable, "bench.py", "--impl", "reference", "--workload", "ctx_b2_q1_kv4096",
                  "--steps", "1", "--warmup", "3", "--ref-rows", "8"])
    assert len(lines) == 1
    _check_line(json.loads(lines[0]), "ctx_b2_q1_kv4096", "TFLOP/s", 1, 3, 1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_torchrun_world2_prints_once():
    pytest.importorskip("torch.distributed.run")
    lines = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                  "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
                  "--impl", "reference", "--gpus", "2", "--workload", "decode_b2_cap256",
                  "--steps", "1", "--warmup", "3"])
    assert len(lines) == 1
    _check_line(json.loads(lines[0]), "decode_b2_cap256", "GB/s", 1, 3, 2)
