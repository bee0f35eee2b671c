"""Multi-GPU runs are independent replicas (the path has no exchange step):
the host logic is checked here with two gloo ranks on the CPU, and the
reference arm under torchrun with two processes."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        from sparse_mla_decode_gb300.replicas import job_rate, rank_seed

        # rank r: 10 ms (rank 0) or 12 ms (rank 1) for 4 steps of 1e6 and 2e6 bytes
        ms, total, rate = job_rate(dist, 10.0 + 2.0 * rank, 1e6 * (rank + 1), 4)
        out.put((rank, ms, total, rate, [rank_seed(1000, rank, r) for r in range(3)]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_all_bytes():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {r[0]: r for r in results}
    for rank in (0, 1):
        _, ms, total, rate, _ = by_rank[rank]
        assert ms == pytest.approx(12.0 / 4) and total == pytest.approx(3e6)
        assert rate == pytest.approx(3e6 / 3e-3 / 1e9)
    seeds = by_rank[0][4] + by_rank[1][4]
    assert len(set(seeds)) == len(seeds)  # every rank draws its own inputs


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--config", "tiny", "--steps", "1", "--warmup", "0"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["cpu_baseline"]["kind"] == "oracle"
