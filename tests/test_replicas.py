"""The benchmark on more than one GPU: the library is built for one-GPU runs
(its paired gathers use cluster multicast, which only a one-GPU run may use),
so the decode arm under torchrun prints one line saying so and runs nothing,
and the reference arm (the CPU oracle) prints one line from rank 0. Both run
here on the CPU as two torchrun processes."""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(*args):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py", *args]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    return [json.loads(l) for l in res.stdout.splitlines() if l.startswith("{")]


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    lines = torchrun("--impl", "reference", "--gpus", "2", "--config", "tiny", "--steps", "1", "--warmup", "0")
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["cpu_baseline"]["kind"] == "oracle"


def test_decode_arm_on_two_gpus_says_it_is_single_gpu_and_runs_nothing():
    lines = torchrun("--gpus", "2", "--steps", "1", "--warmup", "0")
    assert len(lines) == 1
    assert lines[0]["n_gpus"] == 2 and "single-GPU" in lines[0]["unavailable"]
