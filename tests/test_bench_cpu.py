"""The benchmark's reference arm (the CPU oracle timed as it stands) keeps the
JSON-line contract: exactly W untimed and K timed steps, reported as given;
one line from rank 0 under a two-rank launch, the other rank exiting 0
without work. Runs on CPU on the smallest workload, and for the prefill
phases on the MHA shape."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["bench.py", "--impl", "reference", "--workload", "h2o_tiny", "--steps", "3", "--warmup", "3",
        "--cpu-seconds", "1"]


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check(line):
    assert line["impl"] == "reference"
    assert line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1
    assert "3 timed steps after 3 untimed" in line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("h2o")


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable] + ARGS, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check(lines[0])


def test_reference_arm_two_ranks_prints_once():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port)] + ARGS + ["--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check(lines[0])


@pytest.mark.parametrize("phase", ["prefill", "snapkv"])
def test_reference_arm_prefill_phases(phase):
    args = ["bench.py", "--impl", "reference", "--phase", phase, "--workload", "h2o_mha", "--steps", "3",
            "--warmup", "3", "--cpu-seconds", "1"]
    r = subprocess.run([sys.executable] + args, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert "3 timed steps after 3 untimed" in line["cpu_baseline"]["sample"]
    assert line["config"]["prompt_len"] == 2048
