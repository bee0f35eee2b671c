"""Chained multi-layer decode: L back-to-back sparse MLA decode calls per step
(one per layer, each on its own KV rows), captured in a CUDA graph, with and
without programmatic dependent launch (PDL).

    python -m sparse_mla_decode_gb300.chain [--layers 8] [--steps 200] [--shape verify|tiny]

With PDL a layer's kernel is launched while the previous one runs: its set-up
(barrier and TMEM allocation, tensor-map prefetch) overlaps the previous
layer's tail, and it reads its inputs only after its grid-dependency wait. The
module runs itself once per setting (``SMLA_PDL`` is read once per process)
and prints one JSON line per setting and the gain.

Per layer the inputs are one of the seeded single-pool latency workloads
(``verify``: 5 rows x 128 heads x <= 256 keys; ``tiny``: 1 x 16 x 256), with
its rows renumbered into a block of a shared pool of N(0, 1) E4M3 rows;
consecutive steps rotate over blocks (more than 2.5x the L2 in all), so every
layer streams its rows from HBM.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024


def make_sets(shape: str, layers: int, sets: int | None, dev):
    """The chain's inputs: ``sets`` input sets (None: enough that one pass over
    them reads more than 2.5x the L2) of ``layers`` calls each, and the shared
    pool they read. Each call is a dict of device tensors (``q``, ``pools``,
    ``indices``, ``lens``, ``sinks``, ``out``, ``lse``) plus ``w``, its
    workload with the indices renumbered into the shared pool."""
    import numpy as np
    import torch

    from sparse_mla_decode_gb300 import workloads

    make = {"verify": workloads.verify_rows, "tiny": workloads.tiny}[shape]
    ws = [make(seed=5000 + 97 * l) for l in range(layers)]
    # Each (set r, layer l) reads its own block of `block` rows of one pool:
    # the layer's distinct rows are renumbered into the block, so that every
    # step reads rows no other step reads (R steps of rows > 2.5x the L2).
    block = 1024
    uniq = [np.unique(w["indices"][w["indices"] >= 0]) for w in ws]
    assert all(u.size <= block for u in uniq)
    D = ws[0]["q"].shape[2]
    per_step = sum(u.size for u in uniq) * D
    R = sets or int(min(256, max(4, math.ceil(2.5 * L2_BYTES / per_step))))
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    pool = torch.randn((R * layers * block, D), generator=gen, device=dev).to(torch.float8_e4m3fn).view(torch.uint8)
    steps_sets = []
    for r in range(R):
        calls = []
        for l, w in enumerate(ws):
            idx = w["indices"].copy()
            keep = idx >= 0
            idx[keep] = np.searchsorted(uniq[l], idx[keep]) + (r * layers + l) * block
            T, H, _ = w["q"].shape
            calls.append({
                "q": torch.from_numpy(w["q"]).to(dev), "pools": [pool],
                "indices": torch.from_numpy(idx.astype(np.int32)).to(dev),
                "lens": torch.from_numpy(w["lens"]).to(dev),
                "sinks": None if w["sinks"] is None else torch.from_numpy(w["sinks"]).to(dev),
                "out": torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev),
                "lse": torch.empty((T, H), dtype=torch.float32, device=dev),
                "w": dict(w, indices=idx.astype(np.int32)),
            })
        steps_sets.append(calls)
    return pool, steps_sets


def run_layers(calls) -> None:
    """One step: the layers' decode calls, back to back on the current stream."""
    from sparse_mla_decode_gb300 import smla

    for c in calls:
        w = c["w"]
        smla.smla_decode(c["q"], c["pools"], c["indices"], c["lens"], c["sinks"], w["bmm1_scale"],
                         w["bmm2_scale"], w["k_scale"], c["out"], c["lse"], pool_split=w.get("pool_split", 0))


def measure(shape: str, layers: int, steps: int) -> dict:
    import torch

    import __graft_entry__
    from sparse_mla_decode_gb300 import smla

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _, steps_sets = make_sets(shape, layers, None, dev)
    R = len(steps_sets)

    def step(i):
        run_layers(steps_sets[i % R])

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(steps):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    bits = smla.smla_device_error()
    if bits != 0:
        raise RuntimeError(f"device error bits {bits}")
    us_step = e0.elapsed_time(e1) * 1e3 / steps
    return {"shape": shape, "layers": layers, "steps": steps, "input_sets": R,
            "pdl": os.environ.get("SMLA_PDL", "1") != "0",
            "us_per_step": round(us_step, 3), "us_per_layer": round(us_step / layers, 3)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--shape", choices=["verify", "tiny"], default="verify")
    ap.add_argument("--one", action="store_true", help="measure the current SMLA_PDL setting only")
    args = ap.parse_args()
    if args.one:
        print(json.dumps(measure(args.shape, args.layers, args.steps)), flush=True)
        return
    rows = []
    for pdl in ("1", "0"):
        env = dict(os.environ, SMLA_PDL=pdl)
        out = subprocess.run([sys.executable, "-m", "sparse_mla_decode_gb300.chain", "--one", "--layers",
                              str(args.layers), "--steps", str(args.steps), "--shape", args.shape],
                             env=env, cwd=ROOT, capture_output=True, text=True, check=True)
        row = json.loads(out.stdout.strip().splitlines()[-1])
        rows.append(row)
        print(json.dumps(row), flush=True)
    on, off = rows
    print(json.dumps({"shape": args.shape, "layers": args.layers,
                      "pdl_gain_us_per_layer": round(off["us_per_layer"] - on["us_per_layer"], 3),
                      "pdl_speedup": round(off["us_per_step"] / on["us_per_step"], 4)}), flush=True)


if __name__ == "__main__":
    main()
