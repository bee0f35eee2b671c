#!/usr/bin/env python
"""Benchmark: sparse MLA decode on GB300 (µs per call, achieved HBM GB/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config batch|tiny|verify|two_pool|merge|mxfp4|value|merge_value]

A step is one smla_decode call over one batch of seeded synthetic inputs. The
default workload is the bandwidth-bound batch: 64 tokens x 128 heads x 2048
top-k keys of 576-byte E4M3 rows from a 1,048,576-row pool, half of each
token's rows drawn from a shared 20k-row hot set. Inputs are resident in HBM
before timing; consecutive steps rotate over input sets whose distinct rows
sum to more than twice the L2, so each step streams its KV rows from HBM.

One JSON line on rank 0:
  value       algorithmic bytes (unique gathered KV rows + Q + out) / time, GB/s
  ms_per_step device time per call (CUDA events, max over ranks)
  roofline    achieved GB/s of the decode kernel vs the measured HBM copy peak
  e2e         the same metric with host buffers: per step the H2D copy of q,
              indices and lens from pinned memory, the call, and the D2H copy
              of out and lse, all inside the timed region (consecutive steps
              pipelined over three streams)
  cpu_baseline the CPU oracle (fp64 definition) on a bounded sample, all cores
With --impl reference the same line is produced by the CPU oracle alone.
The library is built for runs on one GPU (its paired gathers use cluster
multicast, which only a one-GPU run may use): with --gpus N > 1 or under a
torchrun of several processes, this arm prints one line saying so and runs
nothing. The reference arm (the CPU oracle) runs on rank 0 alone.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


METRIC = "µs/call and achieved HBM GB/s (% of 8 TB/s) for sparse MLA decode"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=["batch", "tiny", "verify", "two_pool", "merge", "mxfp4", "value",
                                         "merge_value", "ds_mla"],
                    default="batch",
                    help="merge: the LSE merge of 8 partial (out, lse) sets of the 64 x 128 batch shape; "
                         "mxfp4: the MXFP4 indexer-query quantisation of 16384 tokens x 32 heads; "
                         "value: the value projection (W_UV) and sigmoid gate of the 64 x 128 batch shape; "
                         "merge_value: the merge of 8 partial sets fused with that projection; "
                         "ds_mla: the 64 x 128 x 2048 batch over 656-byte fp8_ds_mla rows")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work of the oracle baseline sample")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--launch", choices=["graph", "eager"], default="graph",
                    help="time the K calls replayed from one CUDA graph (device time, no host launch "
                         "cost), or as K library calls from Python")
    ap.add_argument("--l2", choices=["rotate", "flush"], default="rotate",
                    help="small workloads: rotate over enough input sets with distinct rows to exceed "
                         "2x L2 (back-to-back calls), or flush L2 before every timed call")
    ap.add_argument("--soak", type=float, default=0.6,
                    help="seconds of untimed calls after the timed region, under the clock sampler")
    return ap.parse_args()


# ------------------------------------------------------------------ inputs


def make_sets(config: str, rank: int, sets: int):
    from sparse_mla_decode_gb300 import workloads

    if config == "batch":
        rng = np.random.default_rng(5000)
        pool = workloads.e4m3_normal(rng, (1 << 20, 576))
        return [workloads.bandwidth_batch(seed=1003 + r, pool=pool) for r in range(sets)]
    make = {"tiny": workloads.tiny, "verify": workloads.verify_rows,
            "two_pool": workloads.two_pool_sinks}[config]
    base = {"tiny": 1000, "verify": 1001, "two_pool": 1002}[config]
    return [make(seed=base + r) for r in range(sets)]


def bytes_alg(w) -> int:
    """Unique gathered KV rows x row bytes + Q + BF16 out (per call)."""
    from sparse_mla_decode_gb300 import workloads

    T, H, D = w["q"].shape
    return workloads.unique_active_rows(w) * D + T * H * D + T * H * 512 * 2


def flops_alg(w) -> int:
    T, H, D = w["q"].shape
    active = 0
    for t in range(T):
        n = max(0, min(int(w["lens"][t]), w["indices"].shape[1]))
        active += int(np.count_nonzero(w["indices"][t, :n] >= 0))
    return active * H * (2 * D + 2 * 512)


def workload_name(config: str, w) -> str:
    T, H, D = w["q"].shape
    W = w["indices"].shape[1]
    desc = {
        "batch": f"{T} tokens x {H} heads x {W} top-k keys, {D}-byte E4M3 rows, 1,048,576-row pool, "
                 "~50% of rows shared via a 20k-row hot set",
        "tiny": f"{T} token x {H} heads x {W} keys, {D}-byte rows, 4096-row pool",
        "verify": f"{T} verify rows x {H} heads x <= {W} keys, {D}-byte rows, k_scale 0.05, one empty row",
        "two_pool": f"{T} tokens x {H} heads, width {W} over two pools (128 window + top-k), "
                    f"{D}-byte rows, sinks",
    }[config]
    return f"{w['name']}: {desc}"


# -------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9 or not (t0 - 0.15 <= ts <= t1 + 0.15):
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, name in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(name)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------- helpers


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {"value": ("smla_value.cu", "smla_ptx.cuh", "smla_merge_row.cuh"),
                  "merge_value": ("smla_value.cu", "smla_ptx.cuh", "smla_merge_row.cuh"),
                  "merge": ("smla_merge.cu", "smla_merge_row.cuh"),
                  "mxfp4": ("smla_quant.cu",),
                  "ds_mla": ("smla_ds_mla.cu", "smla_ptx.cuh")}


def code_text(source: str) -> str:
    """A C++/CUDA source without its comments and with its whitespace runs
    collapsed: what the compiler sees, so that editing a comment does not
    count as changing the kernel. String and character literals are kept as
    they are."""
    out, i, n = [], 0, len(source)
    while i < n:
        ch = source[i]
        if ch in "\"'":
            j = i + 1
            while j < n and source[j] != ch:
                j += 2 if source[j] == "\\" else 1
            out.append(source[i:j + 1])
            i = j + 1
        elif source.startswith("//", i):
            j = source.find("\n", i)
            i = n if j < 0 else j
        elif source.startswith("/*", i):
            j = source.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


def kernel_sha(config: str = "batch") -> str:
    """Hash of the code (comments and whitespace aside) of the sources of the
    kernel a config times (the decode kernel unless listed in KERNEL_SOURCES):
    the committed DRAM traffic holds only while that code is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_mla_decode_gb300", "csrc")
    for name in KERNEL_SOURCES.get(config, ("smla_decode.cu", "smla_ptx.cuh")):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(code_text(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(config: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    entry = data.get(config)
    if not entry or entry.get("kernel_sha") != kernel_sha(config):
        return None
    return entry.get("dram_bytes_per_launch")


def _median_rate(run, n_of, seconds: float, reps: int = 3):
    """Wall-clock median of ``reps`` runs of ``run(n)`` on ``n`` (token, head)
    pairs, ``n`` sized from a probe so that each run takes about ``seconds``.
    Returns (median seconds per pair, n, the runs' seconds)."""
    probe = n_of(None)
    t0 = time.perf_counter()
    run(probe)
    per_pair = (time.perf_counter() - t0) / probe
    n = n_of(int(seconds / max(per_pair, 1e-9)))
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        run(n)
        times.append(time.perf_counter() - t0)
    return float(np.median(times)) / n, n, times


def cpu_oracle_rate(sets, seconds: float):
    """Times the fp64 oracle on bounded samples of (token, head) pairs of the
    first input set: on all host cores and on one core, each the wall-clock
    median of 3 runs. ``seconds`` is the whole CPU budget. Returns the
    cpu_baseline entry (its value: the all-cores rate, GB/s-equivalent)."""
    from oracle import oracle

    w = sets[0]
    T, H = w["q"].shape[:2]
    prob = oracle.Problem.from_workload(w)
    cores = oracle.max_threads()
    rng = np.random.default_rng(11)

    def leg(threads, budget):
        def n_of(n):
            return min(T * H, max(threads, 4) if n is None else max(n, threads, 4))

        def run(n):
            pairs = np.stack([rng.integers(0, T, n), rng.integers(0, H, n)], axis=1)
            oracle.fp64(prob, pairs, threads=threads)

        per_pair, n, times = _median_rate(run, n_of, budget / 3.0)
        per_call = per_pair * T * H
        return {"value": round(bytes_alg(w) / per_call / 1e9, 6), "cores": threads,
                "us_per_call": round(per_call * 1e6, 1),
                "sample": f"{n} of {T * H} (token, head) pairs of one call per run, median of 3 runs "
                          f"({', '.join(f'{t:.2f}' for t in times)} s)"}

    everything = leg(cores, 0.6 * seconds)
    one = leg(1, 0.4 * seconds)
    return {"value": everything["value"], "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": everything["sample"], "us_per_call": everything["us_per_call"],
            "statistic": "wall-clock median of 3 runs, scaled from the sampled pairs to the whole call",
            "one_core": one}


def gather_floor(w, plan):
    """The time the decode's gathers alone need per call, modelled from the
    measured landing rates of profiles/row_gather_peak.json (per SM, cold and
    L2-hot rows, for the gather method the plan uses: paired tile::gather4
    multicast or cp.async; the 7-warp rows, the nearest measured to the
    kernel's 6 producer warps): per (token, head tile, split) CTA,
    its rows that other tokens also read (L2 hits after the first) at the hot
    rate, the others at the cold rate; the slowest CTA of one wave, times the
    number of waves. None when the profile is missing."""
    try:
        with open(os.path.join(ROOT, "profiles", "row_gather_peak.json")) as f:
            rows = json.load(f)["rows"]
    except (OSError, KeyError, ValueError):
        return None
    method = 2 if plan["pair"] == 2 else 0
    rate = {r["pool"]: r["sm_bytes_per_ns"] for r in rows if r["method"] == method and r["issuers"] == 7}
    T, W = w["indices"].shape
    D = w["q"].shape[2]
    seen = {}
    for t in range(T):
        n = max(0, min(int(w["lens"][t]), W))
        for r in set(int(x) for x in w["indices"][t, :n] if x >= 0):
            seen[r] = seen.get(r, 0) + 1
    per_split = plan["chunks_per_split"] * plan["chunk"]
    worst = 0.0
    for t in range(T):
        n = max(0, min(int(w["lens"][t]), W))
        cols = w["indices"][t, :n]
        for sp in range(plan["splits"]):
            part = cols[sp * per_split:(sp + 1) * per_split]
            part = part[part >= 0]
            hot = sum(1 for r in part if seen.get(int(r), 0) > 1)
            ns = (hot * D) / rate["hot"] + ((part.size - hot) * D) / rate["cold"]
            worst = max(worst, ns)
    waves = math.ceil(plan["ctas"] / max(1, plan["resident_ctas"]))
    return {"us": round(worst * waves / 1e3, 2), "method": "paired tile::gather4 multicast" if method == 2 else "cp.async",
            "source": "profiles/row_gather_peak.json"}


def fp8_peak():
    """The dense FP8 tensor peak measured by this library's own tcgen05
    microbenchmark (profiles/fp8_mma_peak.json), else twice the measured BF16
    burst peak."""
    try:
        with open(os.path.join(ROOT, "profiles", "fp8_mma_peak.json")) as f:
            return float(json.load(f)["fp8_dense_peak_tflops"]), "measured (profiles/fp8_mma_peak.json, tcgen05 kind::f8f6f4)"
    except (OSError, KeyError, ValueError):
        pass
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return 2.0 * float(json.load(f)["bf16_tflops"]), "2x the measured BF16 burst peak"
    except (OSError, KeyError, ValueError):
        return 2.0 * 1900.0, "2x the fallback BF16 peak"


# --------------------------------------------------------------- our arm


def pipelined_e2e(torch, host_inputs, dev_like, run, out_like, steps, warmup=3, graph=True):
    """End to end through the library call with host buffers: every step copies
    its inputs from pinned host memory to the device, runs the call, and reads
    its outputs back to pinned host memory. Steps are pipelined over three
    streams and three device slots (the H2D copy of step i + 1 and the D2H copy
    of step i - 1 overlap the call of step i); events order every reuse of a
    slot. With ``graph`` the timed steps (copies included) are captured once in
    a CUDA graph and replayed, so that host launch cost does not bound small
    steps. Returns the mean time per step in ms (CUDA events).

    host_inputs: list (cycled over steps) of tuples of pinned host tensors;
    dev_like: one such tuple on the device (shapes and dtypes of a slot);
    run(inputs, outputs): launches the call on the current stream;
    out_like: tuple of device tensors shaped like the outputs."""
    slots = 3
    d_in = [tuple(torch.empty_like(x) for x in dev_like) for _ in range(slots)]
    d_out = [tuple(torch.empty_like(x) for x in out_like) for _ in range(slots)]
    h_out = [tuple(torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in out_like) for _ in range(slots)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: [torch.cuda.Event() for _ in range(slots)]  # noqa: E731
    e_in, e_comp, e_out = ev(), ev(), ev()

    def issue(first, n):
        comp = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(comp)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        for i in range(first, first + n):
            b = i % slots
            src = host_inputs[i % len(host_inputs)]
            with torch.cuda.stream(s_in):
                if i - first >= slots:
                    s_in.wait_event(e_comp[b])  # the call of step i - 3 has read this slot
                for d, h in zip(d_in[b], src):
                    d.copy_(h, non_blocking=True)
                e_in[b].record(s_in)
            comp.wait_event(e_in[b])
            if i - first >= slots:
                comp.wait_event(e_out[b])  # step i - 3's outputs have left this slot
            run(d_in[b], d_out[b])
            e_comp[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_comp[b])
                for h, d in zip(h_out[b], d_out[b]):
                    h.copy_(d, non_blocking=True)
                e_out[b].record(s_out)
        for s_ in (s_in, s_out):  # join
            e = torch.cuda.Event()
            e.record(s_)
            comp.wait_event(e)

    issue(0, warmup)
    torch.cuda.synchronize()
    comp = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            issue(warmup, steps)
        g.replay()
        torch.cuda.synchronize()
        t0.record(comp)
        g.replay()
        t1.record(comp)
    else:
        t0.record(comp)
        issue(warmup, steps)
        t1.record(comp)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def e2e_entry(torch, step_bytes, host, dev_like, run, out_like, steps, h2d, d2h):
    """The e2e entry: the steps issued eagerly from Python (every step pays the
    API's host work: validation, planning, tensor-map encoding, the ctypes
    call) as the value, and the same steps replayed from one CUDA graph
    beside it."""
    eager = pipelined_e2e(torch, host, dev_like, run, out_like, steps, graph=False)
    graph = pipelined_e2e(torch, host, dev_like, run, out_like, steps, graph=True)
    return {"value": round(step_bytes / (eager * 1e-3) / 1e9, 2), "unit": "GB/s",
            "us_per_call": round(eager * 1e3, 3), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipeline": "per step: H2D of the inputs from pinned memory, the library call, D2H of the outputs to "
                        "pinned memory, on three streams over three slots, issued eagerly from Python",
            "graph": {"value": round(step_bytes / (graph * 1e-3) / 1e9, 2), "unit": "GB/s",
                      "us_per_call": round(graph * 1e3, 3),
                      "pipeline": "the same steps (copies included) captured once in a CUDA graph and replayed"}}


def run_ours(args, rank, world, local_rank):
    import torch

    import __graft_entry__
    from sparse_mla_decode_gb300 import smla

    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    rotate_small = args.config != "batch" and args.l2 == "rotate"
    sets_n = 6 if args.config == "batch" else (1 if rotate_small else 8)
    sets = make_sets(args.config, rank, sets_n)
    pools_dev = {}
    dsets = []
    if rotate_small:
        # One drawn workload replicated R times into pools R times as tall;
        # copy r reads rows shifted by r pool heights, so consecutive calls
        # touch distinct rows and R of them exceed twice the L2.
        w = sets[0]
        per_call = bytes_alg(w)
        R = int(min(4096, max(8, math.ceil(2.5 * L2_BYTES / per_call))))
        T, H, _ = w["q"].shape
        big = [torch.from_numpy(p).to(dev).repeat(R, 1) for p in w["pools"]]
        idx0 = torch.from_numpy(w["indices"]).to(dev)
        W = idx0.shape[1]
        col = torch.arange(W, device=dev)
        rows_of_col = torch.where((len(w["pools"]) == 2) & (col >= w.get("pool_split", 0)),
                                  w["pools"][-1].shape[0], w["pools"][0].shape[0])
        q0 = torch.from_numpy(w["q"]).to(dev)
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        lens = torch.from_numpy(w["lens"]).to(dev)
        sinks = None if w["sinks"] is None else torch.from_numpy(w["sinks"]).to(dev)
        q_all = q0.unsqueeze(0).repeat(R, 1, 1, 1)
        idx_all = torch.where(idx0 >= 0, idx0 + torch.arange(R, device=dev).view(R, 1, 1) * rows_of_col,
                              idx0).to(torch.int32).contiguous()
        for r in range(R):
            dsets.append({"q": q_all[r], "pools": big, "indices": idx_all[r], "lens": lens,
                          "sinks": sinks, "out": out, "lse": lse})
        sets = [w] * R
    else:
        for w in sets:
            key = id(w["pools"][0])
            if key not in pools_dev:
                pools_dev[key] = [torch.from_numpy(p).to(dev) for p in w["pools"]]
            T, H, _ = w["q"].shape
            dsets.append({
                "q": torch.from_numpy(w["q"]).to(dev),
                "pools": pools_dev[key],
                "indices": torch.from_numpy(w["indices"]).to(dev),
                "lens": torch.from_numpy(w["lens"]).to(dev),
                "sinks": None if w["sinks"] is None else torch.from_numpy(w["sinks"]).to(dev),
                "out": torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev),
                "lse": torch.empty((T, H), dtype=torch.float32, device=dev),
            })
    byts = [bytes_alg(sets[0])] * len(sets) if rotate_small else [bytes_alg(w) for w in sets]
    flops = [flops_alg(sets[0])] * len(sets) if rotate_small else [flops_alg(w) for w in sets]
    T, H, D = sets[0]["q"].shape
    shape = smla.make_shape(T, H, sets[0]["indices"].shape[1], D, len(sets[0]["pools"]),
                            sets[0].get("pool_split", 0))
    plan = smla.smla_plan_for(shape)
    stream = torch.cuda.current_stream(dev)
    flush = None if (args.config == "batch" or rotate_small) else torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)

    def call(i):
        w, d = sets[i % len(sets)], dsets[i % len(sets)]
        smla.smla_decode(d["q"], d["pools"], d["indices"], d["lens"], d["sinks"], w["bmm1_scale"],
                         w["bmm2_scale"], w["k_scale"], d["out"], d["lse"], stream=None,
                         pool_split=w.get("pool_split", 0))


    def barrier():
        torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for i in range(max(3, args.warmup)):
        call(i)
    barrier()
    bits = smla.smla_device_error()
    if bits != 0:
        raise RuntimeError(f"device error bits {bits} during warm-up")
    graph = None
    if flush is None and args.launch == "graph":
        # the K timed calls, captured once; the capture stream becomes the
        # current stream inside the context, which the calls launch on
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                call(i)
        graph.replay()
        barrier()
    t_wall0 = time.time()
    if graph is not None:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        graph.replay()
        end.record(stream)
        torch.cuda.synchronize()
        elapsed_ms = start.elapsed_time(end)
    elif flush is None:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            call(i)
        end.record(stream)
        torch.cuda.synchronize()
        elapsed_ms = start.elapsed_time(end)
    else:  # latency workloads: L2 flushed before every timed call
        elapsed_ms = 0.0
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            evs[i][0].record(stream)
            call(i)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        elapsed_ms = sum(a.elapsed_time(b) for a, b in evs)
    t_wall1 = time.time()
    # keep the GPU under the same load for the clock sampler when the timed
    # region was shorter than a few samples
    soak_until = t_wall1 + max(0.0, args.soak - (t_wall1 - t_wall0)) if args.soak > 0 else t_wall1
    i = 0
    while time.time() < soak_until:
        if graph is not None:
            graph.replay()
        else:
            for _ in range(200):
                call(i)
                i += 1
        torch.cuda.synchronize()
    clocks = sampler.stop(t_wall0, max(t_wall1, soak_until))
    bits = smla.smla_device_error()
    if bits != 0:
        raise RuntimeError(f"device error bits {bits} during the timed region")

    step_bytes = float(np.mean([byts[i % len(byts)] for i in range(args.steps)]))
    step_flops = float(np.mean([flops[i % len(flops)] for i in range(args.steps)]))
    ms = elapsed_ms / args.steps
    total_bytes = step_bytes
    value = total_bytes / (ms * 1e-3) / 1e9

    # end to end through the public API, host buffers in pinned memory
    e2e = None
    if not args.no_e2e:
        # q, indices and lens of each input set, resident on the host
        host = [(d["q"].cpu().pin_memory(), d["indices"].cpu().pin_memory(), d["lens"].cpu().pin_memory())
                for d in dsets[:64]]
        h2d = sum(x.numel() * x.element_size() for x in host[0])
        d2h = T * H * 512 * 2 + T * H * 4
        w0 = sets[0]

        def e2e_run(inp, outp):
            q, idx, lens = inp
            smla.smla_decode(q, dsets[0]["pools"], idx, lens, dsets[0]["sinks"], w0["bmm1_scale"],
                             w0["bmm2_scale"], w0["k_scale"], outp[0], outp[1], pool_split=w0.get("pool_split", 0))

        steps = min(args.steps, 500)
        like = ((dsets[0]["q"], dsets[0]["indices"], dsets[0]["lens"]), (dsets[0]["out"], dsets[0]["lse"]))
        e2e = e2e_entry(torch, total_bytes, host, like[0], e2e_run, like[1], steps, h2d, d2h)

    if rank != 0:
        return
    peak, peak_src = measured_hbm_peak()
    achieved = step_bytes / (ms * 1e-3) / 1e9  # this rank's kernel
    traffic = ncu_traffic(args.config)
    cpu = None if args.no_cpu else cpu_oracle_rate(sets, args.cpu_seconds)
    fp8_peak_tflops, fp8_peak_src = fp8_peak()
    floor = gather_floor(sets[0], plan) if args.config == "batch" else None
    if floor is not None:
        floor["frac"] = round(floor["us"] / (ms * 1e3), 4)  # the kernel's time against its gather floor
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 6),
        "us_per_call": round(ms * 1e3, 3),
        "pct_of_8tbs": round(100.0 * achieved / NOMINAL_HBM_GBS, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic",
        "config": {
            "workload": workload_name(args.config, sets[0]),
            "tokens": int(T), "heads": int(H), "width": int(sets[0]["indices"].shape[1]),
            "head_dim": int(D), "input_sets": len(sets),
            "l2": ("rotating %d input sets over distinct rows (~%.2f MB per call, %.0f MB in all) between "
                   "back-to-back calls" % (len(sets), np.mean(byts) / 1e6, np.mean(byts) * len(sets) / 1e6))
                  if flush is None else
                  "L2 flushed (256 MB write) before every timed call",
            "launch": ("one CUDA graph of the %d timed library calls, replayed once" % args.steps)
                      if graph is not None else "%d library calls from Python" % args.steps,
            "plan": plan,
            "parallelism": "single GPU",
        },
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": peak_src,
            "traffic": traffic, "bytes_alg_per_launch": int(step_bytes),
            "tensor_tflops": round(step_flops / (ms * 1e-3) / 1e12, 2),
            "tensor_frac_of_fp8_peak": round(step_flops / (ms * 1e-3) / 1e12 / fp8_peak_tflops, 4),
            "fp8_peak_tflops": fp8_peak_tflops, "fp8_peak_source": fp8_peak_src,
            "gather_floor": floor,
        },
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(args.steps),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------- reference arm


def run_reference(args, rank, world):
    """The CPU oracle (fp64 definition) as the reference implementation; rank 0
    alone runs it. Each step is the oracle over a bounded sample of the call's
    (token, head) pairs (the whole call when it fits), sized so that the
    warm-up and timed steps take about two minutes in all: ``ms_per_step`` is
    the measured time of such a step, and ``value`` the sample's bytes over
    that time (the rate scaled to a whole call, which is what
    ``us_per_call_extrapolated`` states)."""
    if rank != 0:
        return
    from oracle import oracle

    oracle.build()
    sets = make_sets(args.config, 0, 1)
    w = sets[0]
    T, H, D = w["q"].shape
    prob = oracle.Problem.from_workload(w)
    cores = oracle.max_threads()
    rng = np.random.default_rng(13)
    probe = min(T * H, max(cores, 16))
    pairs = np.stack([rng.integers(0, T, probe), rng.integers(0, H, probe)], axis=1)
    t0 = time.perf_counter()
    oracle.fp64(prob, pairs, threads=cores)
    per_pair = (time.perf_counter() - t0) / probe
    total_steps = max(1, args.steps + args.warmup)
    budget = 120.0  # seconds for the whole run
    n = int(max(1, min(T * H, budget / total_steps / max(per_pair, 1e-9))))
    whole = n == T * H
    every = np.stack([np.repeat(np.arange(T), H), np.tile(np.arange(H), T)], axis=1)

    def sample():
        if whole:
            return every
        return np.stack([rng.integers(0, T, n), rng.integers(0, H, n)], axis=1)

    for _ in range(args.warmup):
        oracle.fp64(prob, sample(), threads=cores)
    elapsed = 0.0
    for _ in range(args.steps):
        pairs = sample()
        t0 = time.perf_counter()
        oracle.fp64(prob, pairs, threads=cores)
        elapsed += time.perf_counter() - t0
    step_s = elapsed / args.steps
    per_call = step_s / n * T * H
    value = bytes_alg(w) * (n / (T * H)) / step_s / 1e9
    desc = (f"the whole call ({T * H} (token, head) pairs) per step" if whole else
            f"{n} of {T * H} (token, head) pairs per step, drawn at random")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3),
        "us_per_call_extrapolated": round(per_call * 1e6, 1), "extrapolated": not whole,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": workload_name(args.config, w), "tokens": int(T), "heads": int(H),
                   "width": int(w["indices"].shape[1]), "head_dim": int(D), "step": desc},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


DS_MLA_METRIC = "µs/call and achieved HBM GB/s for sparse MLA decode over 656-byte fp8_ds_mla rows"


def ds_mla_bytes(w) -> int:
    """Unique gathered rows x 656 + Q (512 E4M3 + 64 BF16 per head) + BF16 out."""
    from sparse_mla_decode_gb300 import workloads

    T, H, _ = w["q_latent"].shape
    return workloads.unique_active_rows(w) * 656 + T * H * (512 + 128) + T * H * 512 * 2


def ds_mla_sets(rank: int, sets: int):
    from sparse_mla_decode_gb300 import workloads

    rng = np.random.default_rng(7000 + rank)
    pool = workloads.ds_mla_rows(rng, 1 << 20)
    return [workloads.ds_mla_batch(seed=1007 + r + 100 * rank, pool=pool) for r in range(sets)]


def ds_mla_cpu_rate(w, seconds: float, reps: int = 3):
    """The FP64 definition over fp8_ds_mla rows (numpy) on a bounded sample of
    tokens (all heads each), median of ``reps`` runs; scaled to a whole call."""
    from oracle import ds_mla

    T, H, _ = w["q_latent"].shape
    import torch

    q = torch.cat([torch.from_numpy(w["q_latent"]).view(torch.float8_e4m3fn).to(torch.float64),
                   torch.from_numpy(w["q_rope"].view(np.int16)).view(torch.bfloat16).to(torch.float64)], -1).numpy()
    pool = w["pools"][0]

    def run(n):
        ds_mla.fp64(q[:n], pool, w["indices"][:n], w["lens"][:n], None, w["bmm1_scale"], w["bmm2_scale"])

    t0 = time.perf_counter()
    run(1)
    per_token = time.perf_counter() - t0
    n = int(max(1, min(T, seconds / reps / max(per_token, 1e-9))))
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        run(n)
        times.append(time.perf_counter() - t0)
    per_call = float(np.median(times)) / n * T
    return {"value": round(ds_mla_bytes(w) / per_call / 1e9, 6), "unit": "GB/s", "cores": os.cpu_count(),
            "kind": "oracle", "us_per_call": round(per_call * 1e6, 1), "extrapolated": n < T,
            "sample": f"{n} of {T} tokens (all {H} heads) per run, median of {reps} runs "
                      f"({', '.join(f'{t:.2f}' for t in times)} s); numpy's BLAS threads",
            "statistic": "wall-clock median, scaled from the sampled tokens to the whole call"}


def run_ds_mla(args, rank, world, local_rank):
    """--config ds_mla: smla_decode_ds_mla over the 64 x 128 x 2048 batch of
    656-byte rows, rotating over 6 input sets (distinct rows > 2x L2)."""
    import torch

    import __graft_entry__
    from sparse_mla_decode_gb300 import smla

    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    R = 6
    sets = ds_mla_sets(rank, R)
    pool = torch.from_numpy(sets[0]["pools"][0]).to(dev)
    T, H, _ = sets[0]["q_latent"].shape
    dsets = [{"ql": torch.from_numpy(w["q_latent"]).to(dev),
              "qr": torch.from_numpy(w["q_rope"].view(np.int16)).view(torch.bfloat16).to(dev),
              "idx": torch.from_numpy(w["indices"]).to(dev), "lens": torch.from_numpy(w["lens"]).to(dev),
              "out": torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev),
              "lse": torch.empty((T, H), dtype=torch.float32, device=dev)} for w in sets]
    byts = [ds_mla_bytes(w) for w in sets]
    w0 = sets[0]
    tile = smla.smla_ds_mla_head_tile(T, H)

    def call(i):
        d = dsets[i % R]
        smla.smla_decode_ds_mla(d["ql"], d["qr"], [pool], d["idx"], d["lens"], None, w0["bmm1_scale"],
                                w0["bmm2_scale"], d["out"], d["lse"])

    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for i in range(max(3, args.warmup)):
        call(i)
    torch.cuda.synchronize()
    if smla.smla_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    graph = None
    if args.launch == "graph":
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                call(i)
        graph.replay()
        torch.cuda.synchronize()
    t_wall0 = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            call(i)
    end.record(stream)
    torch.cuda.synchronize()
    elapsed_ms = start.elapsed_time(end)
    t_wall1 = time.time()
    soak_until = t_wall1 + max(0.0, args.soak - (t_wall1 - t_wall0)) if args.soak > 0 else t_wall1
    while time.time() < soak_until:
        if graph is not None:
            graph.replay()
        else:
            for i in range(200):
                call(i)
        torch.cuda.synchronize()
    clocks = sampler.stop(t_wall0, max(t_wall1, soak_until))
    if smla.smla_device_error() != 0:
        raise RuntimeError("device error during the timed region")
    ms = elapsed_ms / args.steps
    per_call = float(np.mean([byts[i % R] for i in range(args.steps)]))
    value = per_call / (ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        host = [(d["ql"].cpu().pin_memory(), d["qr"].cpu().pin_memory(), d["idx"].cpu().pin_memory(),
                 d["lens"].cpu().pin_memory()) for d in dsets]
        h2d = sum(x.numel() * x.element_size() for x in host[0])

        def e2e_run(inp, outp):
            smla.smla_decode_ds_mla(inp[0], inp[1], [pool], inp[2], inp[3], None, w0["bmm1_scale"],
                                    w0["bmm2_scale"], outp[0], outp[1])

        e2e = e2e_entry(torch, per_call, host, (dsets[0]["ql"], dsets[0]["qr"], dsets[0]["idx"], dsets[0]["lens"]),
                        e2e_run, (dsets[0]["out"], dsets[0]["lse"]), min(args.steps, 500), h2d,
                        T * H * (512 * 2 + 4))
    if rank != 0:
        return
    cpu = None if args.no_cpu else ds_mla_cpu_rate(w0, args.cpu_seconds)
    peak, peak_src = measured_hbm_peak()
    line = {
        "metric": DS_MLA_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "us_per_call": round(ms * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/bf16", "data": "synthetic",
        "config": {"workload": f"{w0['name']}: {T} tokens x {H} heads x 2048 top-k keys, 656-byte fp8_ds_mla rows "
                               "(E4M3 latents, FP32 block scales, BF16 rope), 1,048,576-row pool, ~50% of rows "
                               "shared via a 20k-row hot set",
                   "tokens": T, "heads": H, "width": 2048, "row_bytes": 656, "input_sets": R,
                   "l2": "rotating %d input sets over distinct rows (~%.2f MB per call) between back-to-back calls"
                         % (R, per_call / 1e6),
                   "launch": ("one CUDA graph of the %d timed library calls, replayed once" % args.steps)
                             if graph is not None else "%d library calls from Python" % args.steps,
                   "kernel": "%d-head tiles, one CTA per (token, %d heads): %d CTAs, 128-key chunks in two stages"
                             % (tile, tile, T * H // tile),
                   "parallelism": "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(value, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(value / peak, 4), "peak_source": peak_src, "traffic": ncu_traffic("ds_mla"),
                     "bytes_alg_per_launch": int(per_call)},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(args.steps), "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def run_ds_mla_reference(args, rank, world):
    """The FP64 definition over fp8_ds_mla rows as the reference arm (rank 0)."""
    if rank != 0:
        return
    w = ds_mla_sets(0, 1)[0]
    budget = min(120.0, max(5.0, 120.0 / max(1, args.steps + args.warmup)))
    cpu = ds_mla_cpu_rate(w, budget)
    T, H, _ = w["q_latent"].shape
    line = {
        "metric": DS_MLA_METRIC, "value": cpu["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(cpu["us_per_call"] / 1e3, 3), "extrapolated": cpu["extrapolated"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": w["name"], "tokens": T, "heads": H, "width": 2048, "row_bytes": 656},
        "cpu_baseline": cpu,
        "e2e": {"value": cpu["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


MERGE_METRIC = "µs/call and achieved HBM GB/s for the LSE merge of partial (out, lse) sets"


def merge_bytes(S, T, H) -> int:
    """Bytes of one merge that reads every source row: every source row and LSE
    read once, the merged row and LSE written once (an upper bound, used to
    size the input rotation)."""
    return S * T * H * (512 * 2 + 4) + T * H * (512 * 2 + 4) + T * 4


def merge_bytes_live(lses, lens) -> int:
    """Algorithmic bytes of one merge of these sets: the rows of the sources
    that carry weight (finite LSE, token count > 0) and every LSE read once,
    the merged row and LSE written once. A source without weight needs no row."""
    import torch

    S, T, H = lses.shape
    live = torch.isfinite(lses) & (lens > 0).view(1, T, 1)
    return int(live.sum().item()) * 512 * 2 + S * T * H * 4 + T * H * (512 * 2 + 4) + T * 4


def run_merge(args, rank, world, local_rank):
    """--config merge: smla_merge of 8 partial sets of the 64 x 128 batch shape,
    rotating over input sets whose bytes exceed 2.5x the L2."""
    import torch

    import __graft_entry__
    from sparse_mla_decode_gb300 import smla, workloads

    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    S, T, H = 8, 64, 128
    R = int(math.ceil(2.5 * L2_BYTES / merge_bytes(S, T, H)))
    sets = [workloads.merge_sets(1005 + 17 * r + 1000 * rank, S, T, H, device=dev) for r in range(R)]
    per_call = sum(merge_bytes_live(l, n) for _, l, n in sets) / R  # the sets' mean
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)

    def call(i):
        parts, lses, lens = sets[i % R]
        smla.smla_merge(parts, lses, lens, out, lse)


    def barrier():
        torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for i in range(max(3, args.warmup)):
        call(i)
    barrier()
    graph = None
    if args.launch == "graph":
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                call(i)
        graph.replay()
        barrier()
    t_wall0 = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            call(i)
    end.record(stream)
    torch.cuda.synchronize()
    elapsed_ms = start.elapsed_time(end)
    t_wall1 = time.time()
    soak_until = t_wall1 + max(0.0, args.soak - (t_wall1 - t_wall0)) if args.soak > 0 else t_wall1
    while time.time() < soak_until:
        if graph is not None:
            graph.replay()
        else:
            for i in range(200):
                call(i)
        torch.cuda.synchronize()
    clocks = sampler.stop(t_wall0, max(t_wall1, soak_until))
    ms = elapsed_ms / args.steps
    total_bytes = per_call
    value = total_bytes / (ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        host = [(sets[k][0].cpu().pin_memory(), sets[k][1].cpu().pin_memory()) for k in range(R)]
        h2d = sum(x.numel() * x.element_size() for x in host[0])

        def e2e_run(inp, outp):
            smla.smla_merge(inp[0], inp[1], sets[0][2], outp[0], outp[1])

        e2e = e2e_entry(torch, total_bytes, host, (sets[0][0], sets[0][1]), e2e_run, (out, lse),
                        min(args.steps, 200), h2d, T * H * (512 * 2 + 4))
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu:
        cpu = merge_cpu_rate(sets[0], args.cpu_seconds)
    peak, peak_src = measured_hbm_peak()
    achieved = per_call / (ms * 1e-3) / 1e9
    line = {
        "metric": MERGE_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "us_per_call": round(ms * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16/f32", "data": "synthetic",
        "config": {"workload": f"merge_s{S}_t{T}_h{H}: {S} partial (BF16 [T, H, 512], base-2 LSE) sets of "
                               f"the {T} x {H} batch shape, 3% empty sources, one count-0 token",
                   "sources": S, "tokens": T, "heads": H, "input_sets": R,
                   "l2": "rotating %d input sets (%.1f MB per call, %.0f MB in all) between back-to-back calls"
                         % (R, per_call / 1e6, R * per_call / 1e6),
                   "launch": ("one CUDA graph of the %d timed library calls, replayed once" % args.steps)
                             if graph is not None else "%d library calls from Python" % args.steps,
                   "parallelism": "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src, "traffic": ncu_traffic("merge"),
                     "bytes_alg_per_launch": int(per_call)},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(args.steps), "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def merge_cpu_rate(first_set, seconds: float):
    """The oracle's merge on all host cores over a bounded sample of rows."""
    from oracle import oracle

    oracle.build()
    parts, lses, lens = (x.cpu() for x in first_set)
    S, T, H, _ = parts.shape
    prob = oracle.MergeProblem(parts.view(torch_int16()).numpy().view(np.uint16), lses.numpy(), lens.numpy())
    cores = oracle.max_threads()
    rng = np.random.default_rng(11)
    n = min(T * H, 256)
    t0 = time.perf_counter()
    done = 0
    while time.perf_counter() - t0 < seconds and done < 64 * T * H:
        rows = rng.integers(0, T * H, n)
        oracle.merge(prob, np.stack([rows // H, rows % H], 1), threads=cores)
        done += n
    elapsed = time.perf_counter() - t0
    per_call = elapsed / done * T * H
    return {"value": round(merge_bytes_live(lses, lens) / per_call / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle", "sample": f"{done} merged rows in batches of {n} drawn from the {T * H} rows of one call",
            "us_per_call": round(per_call * 1e6, 1)}


MXFP4_METRIC = "µs/call and achieved HBM GB/s for the MXFP4 indexer-query quantisation"


def mxfp4_bytes(T, H) -> int:
    """BF16 query and FP32 weights read; packed codes, scales and weights written."""
    return T * H * (128 * 2 + 4) + T * H * (64 + 4 + 4)


def run_mxfp4(args, rank, world, local_rank):
    """--config mxfp4: smla_mxfp4_q_quant of a BF16 query [16384, 32, 128]."""
    import torch

    import __graft_entry__
    from sparse_mla_decode_gb300 import smla

    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    T, H = 16384, 32
    per_call = mxfp4_bytes(T, H)
    R = max(2, int(math.ceil(2.5 * L2_BYTES / per_call)))
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242 + rank)
    sets = [(torch.randn((T, H, 128), generator=gen, device=dev).to(torch.bfloat16),
             torch.randn((T, H), generator=gen, device=dev)) for _ in range(R)]
    outs = [(torch.empty((T, H, 64), dtype=torch.uint8, device=dev), torch.empty((T, H), dtype=torch.int32, device=dev),
             torch.empty((T, H), dtype=torch.float32, device=dev)) for _ in range(R)]

    def call(i):
        q, w = sets[i % R]
        smla.smla_mxfp4_q_quant(q, w, 0.0625, *outs[i % R])

    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for i in range(max(3, args.warmup)):
        call(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(args.steps):
            call(i)
    graph.replay()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    while time.time() < t_wall0 + args.soak:
        graph.replay()
        torch.cuda.synchronize()
    clocks = sampler.stop(t_wall0, max(t_wall1, t_wall0 + args.soak))
    ms = start.elapsed_time(end) / args.steps
    achieved = per_call / (ms * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        host = [(sets[k][0].cpu().pin_memory(), sets[k][1].cpu().pin_memory()) for k in range(R)]

        def e2e_run(inp, outp):
            smla.smla_mxfp4_q_quant(inp[0], inp[1], 0.0625, *outp)

        e2e = e2e_entry(torch, per_call, host, sets[0], e2e_run, outs[0], min(args.steps, 100),
                        T * H * (256 + 4), T * H * 72)
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu:
        cpu = mxfp4_cpu_rate(sets[0], args.cpu_seconds)
    peak, peak_src = measured_hbm_peak()
    line = {
        "metric": MXFP4_METRIC, "value": round(per_call * world / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "us_per_call": round(ms * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16->e2m1", "data": "synthetic",
        "config": {"workload": f"mxfp4_q_t{T}_h{H}_d128: BF16 query N(0, 1), FP32 weights",
                   "tokens": T, "heads": H, "head_dim": 128, "input_sets": R,
                   "l2": "rotating %d input sets (%.1f MB per call)" % (R, per_call / 1e6),
                   "launch": "one CUDA graph of the %d timed library calls, replayed once" % args.steps,
                   "pages_context": "the pages' Triton kernel: ~35 us at 16K tokens x 32 heads on GB300"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src, "traffic": ncu_traffic("mxfp4"),
                     "bytes_alg_per_launch": int(per_call)},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(args.steps), "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def mxfp4_cpu_rate(first_set, seconds: float):
    """The oracle's quantisation on the host (one thread per call) over a
    bounded sample of tokens."""
    from oracle import oracle

    oracle.build()
    q, w = (x.cpu() for x in first_set)
    T, H, _ = q.shape
    qf = q.float().numpy()
    wf = w.numpy()
    rng = np.random.default_rng(3)
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds and done < T:
        rows = rng.integers(0, T, 64)
        oracle.mxfp4_q_quant(qf[rows], wf[rows], 0.0625, H)
        done += 64
    per_call = (time.perf_counter() - t0) / done * T
    return {"value": round(mxfp4_bytes(T, H) / per_call / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of {T} tokens in batches of 64", "us_per_call": round(per_call * 1e6, 1)}


def run_mxfp4_reference(args, rank, world):
    if rank != 0:
        return
    import torch

    T, H = 16384, 32
    gen = torch.Generator()
    gen.manual_seed(4242)
    first = (torch.randn((T, H, 128), generator=gen).to(torch.bfloat16), torch.randn((T, H), generator=gen))
    total = max(1, args.steps + args.warmup)
    cpu = mxfp4_cpu_rate(first, min(60.0, 2.0 * total) / total * args.steps)
    line = {
        "metric": MXFP4_METRIC, "value": cpu["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(cpu["us_per_call"] / 1e3, 3), "us_per_call": cpu["us_per_call"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "impl": "reference", "config": {"workload": f"mxfp4_q_t{T}_h{H}_d128", "tokens": T, "heads": H},
        "cpu_baseline": cpu,
        "e2e": {"value": cpu["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


VALUE_METRIC = "µs/call and achieved HBM GB/s for the value projection (W_UV) and sigmoid gate"
MERGE_VALUE_METRIC = ("µs/call and achieved HBM GB/s for the LSE merge of partial sets fused with the value "
                      "projection (W_UV) and sigmoid gate")


def value_bytes(T, H) -> int:
    """Merged BF16 rows, the BF16 W_UV of every head and the BF16 gates read;
    BF16 values written (lens: 4 bytes a token)."""
    return T * H * 512 * 2 + H * 512 * 128 * 2 + 2 * T * H * 128 * 2 + 4 * T


def value_sets(T, H, R, seed, device):
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    sets = []
    for _ in range(R):
        latent = torch.randn((T, H, 512), generator=gen, device=device).to(torch.bfloat16)
        w = (torch.randn((H, 512, 128), generator=gen, device=device) / 512 ** 0.5).to(torch.bfloat16)
        gate = (2.0 * torch.randn((T, H * 128), generator=gen, device=device)).to(torch.bfloat16)
        lens = torch.full((T,), 2048, dtype=torch.int32, device=device)
        sets.append((latent, w, gate, lens))
    return sets


def merge_value_bytes(S, T, H) -> int:
    """Every partial row and LSE, W_UV and the gates read; the values written
    (an upper bound, used to size the input rotation)."""
    return S * T * H * (512 * 2 + 4) + H * 512 * 128 * 2 + 2 * T * H * 128 * 2 + 4 * T


def merge_value_bytes_live(lses, lens) -> int:
    """Algorithmic bytes of one fused merge + projection: the rows of the
    sources that carry weight and every LSE, W_UV and the gates read; the
    values written. (The kernel's TMA boxes also read the rows of empty
    sources, which shows in its DRAM traffic.)"""
    S, T, H = lses.shape
    rows = merge_bytes_live(lses, lens) - S * T * H * 4 - T * H * (512 * 2 + 4) - T * 4
    return rows + S * T * H * 4 + H * 512 * 128 * 2 + 2 * T * H * 128 * 2 + 4 * T


def run_value(args, rank, world, local_rank, fused=False):
    """--config value: smla_value_gate of the 64 x 128 batch shape (one W_UV
    per input set, as for consecutive layers). --config merge_value:
    smla_merge_value of 8 partial sets of that shape."""
    import torch

    import __graft_entry__
    from sparse_mla_decode_gb300 import smla, workloads

    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    S, T, H = 8, 64, 128
    per_call = merge_value_bytes(S, T, H) if fused else value_bytes(T, H)
    R = max(2, int(math.ceil(2.5 * L2_BYTES / per_call)))
    sets = value_sets(T, H, R, 5151 + rank, dev)
    if fused:
        merged = [workloads.merge_sets(1005 + 17 * r + 1000 * rank, S, T, H, device=dev) for r in range(R)]
        sets = [(m[0], m[1], m[2], v[1], v[2]) for m, v in zip(merged, sets)]  # parts, lses, lens, w_uv, gate
        per_call = sum(merge_value_bytes_live(m[1], m[2]) for m in merged) / R  # the sets' mean
    outs = [torch.empty((T, H * 128), dtype=torch.bfloat16, device=dev) for _ in range(R)]

    def call(i):
        if fused:
            parts, lses, lens, w, gate = sets[i % R]
            smla.smla_merge_value(parts, lses, lens, w, gate, outs[i % R])
        else:
            smla.smla_value_gate(*sets[i % R], outs[i % R])

    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for i in range(max(3, args.warmup)):
        call(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(args.steps):
            call(i)
    graph.replay()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    while time.time() < t_wall0 + args.soak:
        graph.replay()
        torch.cuda.synchronize()
    clocks = sampler.stop(t_wall0, max(t_wall1, t_wall0 + args.soak))
    if smla.smla_device_error() != 0:
        raise RuntimeError("value kernel reported a device error")
    ms = start.elapsed_time(end) / args.steps
    achieved = per_call / (ms * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        # the weights stay resident (a layer's W_UV does not travel per call);
        # the rows (or partial sets), gates and counts go up, the values come back
        if fused:
            host = [(sets[k][0].cpu().pin_memory(), sets[k][1].cpu().pin_memory(), sets[k][2].cpu().pin_memory(),
                     sets[k][4].cpu().pin_memory()) for k in range(R)]
            dev_like = (sets[0][0], sets[0][1], sets[0][2], sets[0][4])

            def e2e_run(inp, outp):
                smla.smla_merge_value(inp[0], inp[1], inp[2], sets[0][3], inp[3], outp[0])

            h2d = S * T * H * (512 * 2 + 4) + T * H * 256 + 4 * T
        else:
            host = [(sets[k][0].cpu().pin_memory(), sets[k][2].cpu().pin_memory(), sets[k][3].cpu().pin_memory())
                    for k in range(R)]
            dev_like = (sets[0][0], sets[0][2], sets[0][3])

            def e2e_run(inp, outp):
                smla.smla_value_gate(inp[0], sets[0][1], inp[1], inp[2], outp[0])

            h2d = T * H * 512 * 2 + T * H * 256 + 4 * T
        e2e = e2e_entry(torch, per_call, host, dev_like, e2e_run, (outs[0],), min(args.steps, 100), h2d,
                        T * H * 256)
        e2e["resident"] = "W_UV (a layer's weights do not travel per call)"
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu:
        cpu = value_cpu_rate(sets[0], args.cpu_seconds, fused)
    peak, peak_src = measured_hbm_peak()
    config = "merge_value" if fused else "value"
    if fused:
        workload = (f"merge_value_s{S}_t{T}_h{H}: 8 partial sets (BF16 rows N(0, 1), base-2 LSEs with empty "
                    f"sources), W_UV N(0, 1/512), gates N(0, 4)")
        shape = {"sources": S, "tokens": T, "heads": H, "latent": 512, "values": 128}
    else:
        workload = f"value_gate_t{T}_h{H}: merged BF16 rows N(0, 1), W_UV N(0, 1/512), gates N(0, 4)"
        shape = {"tokens": T, "heads": H, "latent": 512, "values": 128}
    line = {
        "metric": MERGE_VALUE_METRIC if fused else VALUE_METRIC,
        "value": round(per_call * world / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "us_per_call": round(ms * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload, **shape, "input_sets": R,
                   "l2": "rotating %d input sets, W_UV included (%.1f MB per call)" % (R, per_call / 1e6),
                   "launch": "one CUDA graph of the %d timed library calls, replayed once" % args.steps},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src, "traffic": ncu_traffic(config),
                     "bytes_alg_per_launch": int(per_call)},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(args.steps), "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def value_cpu_rate(first_set, seconds: float, fused=False):
    """The oracle's projection and gate (after its merge, when fused) on the
    host over a bounded sample of tokens."""
    from oracle import oracle

    oracle.build()
    if fused:
        parts, lses, lens, w, gate = (x.cpu() for x in first_set)
        S, T, H, _ = parts.shape
        p_b = parts.view(torch_int16()).numpy().view(np.uint16)
    else:
        latent, w, gate, lens = (x.cpu() for x in first_set)
        T, H, _ = latent.shape
        lat_b = latent.view(torch_int16()).numpy().view(np.uint16)
    w_b = w.view(torch_int16()).numpy().view(np.uint16)
    g_b = gate.view(torch_int16()).numpy().view(np.uint16)
    rng = np.random.default_rng(4)
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds and done < T:
        rows = rng.integers(0, T, 2)
        if fused:
            _, m_bits, _ = oracle.merge(oracle.MergeProblem(p_b[:, rows], lses.numpy()[:, rows],
                                                            lens.numpy()[rows]), threads=oracle.max_threads())
            oracle.value_gate(m_bits.reshape(2, H, 512), w_b, g_b[rows], lens.numpy()[rows])
        else:
            oracle.value_gate(lat_b[rows], w_b, g_b[rows], lens.numpy()[rows])
        done += 2
    per_call = (time.perf_counter() - t0) / done * T
    total = merge_value_bytes_live(lses, lens) if fused else value_bytes(T, H)
    return {"value": round(total / per_call / 1e9, 6), "unit": "GB/s", "cores": oracle.max_threads() if fused else 1,
            "kind": "oracle", "sample": f"{done} of {T} tokens, all heads, in batches of 2",
            "us_per_call": round(per_call * 1e6, 1)}


def run_value_reference(args, rank, world, fused=False):
    if rank != 0:
        return
    from sparse_mla_decode_gb300 import workloads

    S, T, H = 8, 64, 128
    first = value_sets(T, H, 1, 5151, "cpu")[0]
    if fused:
        m = workloads.merge_sets(1005, S, T, H)
        first = (m[0], m[1], m[2], first[1], first[2])
    total = max(1, args.steps + args.warmup)
    cpu = value_cpu_rate(first, min(60.0, 2.0 * total) / total * args.steps, fused)
    name = f"merge_value_s{S}_t{T}_h{H}" if fused else f"value_gate_t{T}_h{H}"
    line = {
        "metric": MERGE_VALUE_METRIC if fused else VALUE_METRIC, "value": cpu["value"], "unit": "GB/s",
        "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(cpu["us_per_call"] / 1e3, 3), "us_per_call": cpu["us_per_call"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference", "config": {"workload": name, "tokens": T, "heads": H, **({"sources": S} if fused else {})},
        "cpu_baseline": cpu,
        "e2e": {"value": cpu["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def torch_int16():
    import torch

    return torch.int16


def run_merge_reference(args, rank, world):
    """The oracle's merge as the reference arm; rank 0 alone, bounded samples."""
    if rank != 0:
        return
    from sparse_mla_decode_gb300 import workloads

    S, T, H = 8, 64, 128
    total = max(1, args.steps + args.warmup)
    cpu = merge_cpu_rate(workloads.merge_sets(1005, S, T, H), min(60.0, 2.0 * total) / total * args.steps)
    line = {
        "metric": MERGE_METRIC, "value": cpu["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(cpu["us_per_call"] / 1e3, 3),
        "us_per_call": cpu["us_per_call"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": f"merge_s{S}_t{T}_h{H}", "sources": S, "tokens": T, "heads": H},
        "cpu_baseline": cpu,
        "e2e": {"value": cpu["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if args.config == "merge":
            run_merge_reference(args, rank, world)
        elif args.config == "mxfp4":
            run_mxfp4_reference(args, rank, world)
        elif args.config in ("value", "merge_value"):
            run_value_reference(args, rank, world, fused=args.config == "merge_value")
        elif args.config == "ds_mla":
            run_ds_mla_reference(args, rank, world)
        else:
            run_reference(args, rank, world)
        return
    n_gpus = max(world, args.gpus)
    if n_gpus > 1:
        # one GPU per run: the paired gathers use cluster multicast, which only
        # a run on one GPU may use, so this build has no multi-GPU path
        if rank == 0:
            print(json.dumps({"metric": METRIC, "impl": "ours", "n_gpus": n_gpus,
                              "unavailable": "single-GPU build: its paired gathers use cluster multicast, which "
                                             "only a one-GPU run may use; run with --gpus 1"}), flush=True)
        return
    if args.config == "merge":
        run_merge(args, rank, world, local_rank)
    elif args.config == "mxfp4":
        run_mxfp4(args, rank, world, local_rank)
    elif args.config in ("value", "merge_value"):
        run_value(args, rank, world, local_rank, fused=args.config == "merge_value")
    elif args.config == "ds_mla":
        run_ds_mla(args, rank, world, local_rank)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
