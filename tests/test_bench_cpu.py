"""The benchmark's reference arm (the fp64 oracle timed on the host cores) on
CPU: one JSON line with the contract's keys, printed by rank 0 alone when
launched as several ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _json_lines(stdout: str):
    return [json.loads(l) for l in stdout.splitlines() if l.startswith("{")]


def _check_line(d, n_gpus):
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["n_gpus"] == n_gpus and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "prefill_256k_bf16_b1_l262144_d8192"
    assert d["config"]["calls_per_step"] == 64
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # a step is the bounded sample actually timed: ms_per_step is its time
    # and the value its rate, so steps x ms_per_step is the time really spent
    assert 0 < d["elements_per_step"] < d["config"]["batch"] * d["config"]["seqlen"] * d["config"]["d_inner"]
    assert d["ms_per_step"] == pytest.approx(d["elements_per_step"] / d["value"] * 1e3)
    assert d["ms_per_step"] < 60e3


@pytest.mark.timeout(300)
def test_reference_arm_one_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1)


@pytest.mark.timeout(300)
def test_reference_arm_two_ranks_rank0_prints():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
                        "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 2)
