"""Sweep of sparse MLA decode over tokens x heads x top-k.

    python -m sparse_mla_decode_gb300.sweep [--quick] [--steps K] [--out FILE]

Grid: tokens {1, 2, 6, 12, 32, 128, 256} x heads {16, 64, 128} x top-k
{256, 512, 1024, 2048}. Rows are 576-byte E4M3 N(0, 1) in a 1,048,576-row pool,
indices unique and uniform per token, 10% set to -1, per-token counts uniform
in [k/2, k]. Inputs are drawn on the GPU from seeded torch generators (the same
distributions as ``workloads.sweep_point``); each point rotates over enough
index sets that their distinct rows exceed twice the L2, timed as back-to-back
calls with CUDA events, both eagerly from Python and replayed from a CUDA
graph that holds the same calls (the device time without host launch cost;
``us_per_call``). Reports µs per call, GB/s of algorithmic bytes (unique
active rows + Q + out), the split count the planner chose, and TFLOP/s.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_mla_decode_gb300 import smla  # noqa: E402

TOKENS = (1, 2, 6, 12, 32, 128, 256)
HEADS = (16, 64, 128)
TOPK = (256, 512, 1024, 2048)
POOL_ROWS = 1 << 20
D = 576
L2_BYTES = 129 * 1024 * 1024


def e4m3_normal(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device).to(torch.float8_e4m3fn).view(torch.uint8)


def index_sets(T, k, R, gen, device):
    """R index sets [T, k]: unique uniform rows per token, 10% holes, counts in [k/2, k]."""
    idx = torch.empty((R, T, k), dtype=torch.int32, device=device)
    for r in range(R):
        for t in range(T):
            idx[r, t] = torch.randperm(POOL_ROWS, generator=gen, device=device)[:k].to(torch.int32)
    holes = torch.rand((R, T, k), generator=gen, device=device) < 0.10
    idx[holes] = -1
    lens = torch.randint(k // 2, k + 1, (R, T), generator=gen, device=device, dtype=torch.int32)
    return idx, lens


def point(T, H, k, pool, steps, device, seed, scan=(), tiles=()):
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    per_call = T * 0.9 * 0.75 * k * D
    R = int(min(4096, max(1, math.ceil(2.5 * L2_BYTES / per_call))))
    R = min(R, max(1, 4096 // T))
    q = e4m3_normal((R, T, H, D), gen, device)
    idx, lens = index_sets(T, k, R, gen, device)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((T, H), dtype=torch.float32, device=device)
    # algorithmic bytes and FLOPs, averaged over the sets
    col = torch.arange(k, device=device).view(1, 1, k)
    active = (col < lens.unsqueeze(-1)) & (idx >= 0)
    uniq = 0
    for r in range(R):
        uniq += torch.unique(idx[r][active[r]]).numel()
    bytes_alg = uniq / R * D + T * H * D + T * H * 512 * 2
    flops = active.sum().item() / R * H * (2 * D + 2 * 512)
    bmm1 = 1.0 / math.sqrt(192.0)
    views = [(q[r], idx[r], lens[r]) for r in range(R)]

    def call(i):
        qv, iv, lv = views[i % R]
        smla.smla_decode(qv, [pool], iv, lv, None, bmm1, 1.0, 1.0, out, lse)

    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(eager):
        for i in range(5):
            call(i)
        torch.cuda.synchronize()
        us_eager = None
        if eager:  # one library call per step from Python, back to back
            e0.record(stream)
            for i in range(steps):
                call(i)
            e1.record(stream)
            torch.cuda.synchronize()
            us_eager = e0.elapsed_time(e1) * 1e3 / steps
        # the same calls captured once in a CUDA graph and replayed: device
        # time without the host's launch cost
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(steps):
                call(i)
        graph.replay()
        torch.cuda.synchronize()
        reps = 3
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        del graph
        return e0.elapsed_time(e1) * 1e3 / (steps * reps), us_eager

    us, us_eager = timed(True)
    by_tile = {}
    for n in tiles:
        os.environ["SMLA_HEAD_TILE"] = str(n)
        try:
            pl = smla.smla_plan_for(smla.make_shape(T, H, k, D))
            if pl["head_tile"] == n:
                by_tile[n] = [round(timed(False)[0], 3), pl["splits"]]
        finally:
            del os.environ["SMLA_HEAD_TILE"]
    by_splits = {}
    for s in scan:
        os.environ["SMLA_SPLITS"] = str(s)
        try:
            got = smla.smla_plan_for(smla.make_shape(T, H, k, D))["splits"]
            if got == s:
                by_splits[s] = round(timed(False)[0], 3)
        finally:
            del os.environ["SMLA_SPLITS"]
    bits = smla.smla_device_error()
    plan = smla.smla_plan_for(smla.make_shape(T, H, k, D))
    return {"tokens": T, "heads": H, "topk": k, "us_per_call": round(us, 3), "us_eager": round(us_eager, 3),
            "gbs": round(bytes_alg / (us * 1e-6) / 1e9, 1), "tflops": round(flops / (us * 1e-6) / 1e12, 1),
            "splits": plan["splits"], "ctas": plan["ctas"], "resident_ctas": plan["resident_ctas"], "input_sets": R, "device_error": bits,
            "head_tile": plan["head_tile"],
            **({"us_by_splits": by_splits} if scan else {}),
            **({"us_splits_by_head_tile": by_tile} if tiles else {})}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--quick", action="store_true", help="a corner subset of the grid")
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--out", default=None, help="write the rows as JSON lines here")
    ap.add_argument("--scan-splits", default="", help="also time these forced split counts, e.g. 1,2,4,8")
    ap.add_argument("--scan-tiles", default="", help="also time these forced head tiles, e.g. 16,32,64")
    ap.add_argument("--points", default="", help="only these points, e.g. 1x16x256,64x128x2048")
    args = ap.parse_args()
    import __graft_entry__

    __graft_entry__.build()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(2000)
    pool = e4m3_normal((POOL_ROWS, D), gen, device)
    points = [(t, h, k) for t in TOKENS for h in HEADS for k in TOPK]
    if args.points:
        points = [tuple(int(v) for v in p.split("x")) for p in args.points.split(",")]
    if args.quick:
        points = [p for p in points if p[0] in (1, 12, 256) and p[2] in (256, 2048)]
    rows = []
    for i, (t, h, k) in enumerate(points):
        scan = tuple(int(v) for v in args.scan_splits.split(",") if v)
        tiles = tuple(int(v) for v in args.scan_tiles.split(",") if v)
        row = point(t, h, k, pool, args.steps, device, seed=2000 + 7919 * t + 104729 * h + k, scan=scan,
                    tiles=tiles)
        rows.append(row)
        print(json.dumps(row), flush=True)
        if row["device_error"] != 0:
            raise RuntimeError(f"device error at {row}")
    if args.out:
        with open(args.out, "w") as f:
            for row in rows:
                f.write(json.dumps(row) + "\n")


if __name__ == "__main__":
    main()
