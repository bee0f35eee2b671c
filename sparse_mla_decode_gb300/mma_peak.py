"""FP8 tensor-core rates of this GPU, measured with the library's own tcgen05
microbenchmark (``libsmla_peak.so``, built from ``csrc/smla_peak.cu``).

    python -m sparse_mla_decode_gb300.mma_peak [--json PATH]

For each MMA shape the decode uses or could use (cta_group::1 at M = 128 and
cta_group::2 at M = 256 over a CTA pair; N = 16 / 32 / 64 / 128 / 256; operands K-major
or MN-major as the decode reads them), two numbers:

* ``cycles_per_mma``: one CTA (or pair) issues 4000 K = 32 MMAs into one
  accumulator; the clock64 span from the first issue to the commit's arrival,
  divided by the MMA count. An ideal dense FP8 tensor core does M_cta x N x 32
  multiply-adds in M_cta x N x 32 / 8192 cycles (128 x N x 32 / 8192 = N / 2).
* ``tflops``: every SM does the same; FLOPs of the launch / its CUDA-event time.

A second table takes 2 or 4 accumulators in turn (independent chains) for the
narrow shapes, to tell a per-instruction cost from a chain's serialisation.

The largest ``tflops`` is the measured dense FP8 peak that ``bench.py`` quotes
the decode's tensor fraction against. With ``--json`` the table is written as
JSON (the summary committed under ``profiles/``).
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))

# (cta_group, N, A MN-major, B MN-major, what the decode uses it for)
SHAPES = [
    (1, 16, 0, 0, "QK of a 16-head tile"),
    (1, 16, 1, 1, "PV of a 16-head tile"),
    (1, 32, 0, 0, "QK of a 32-head tile"),
    (1, 32, 1, 1, "PV of a 32-head tile"),
    (1, 64, 0, 0, "QK of a 64-head tile (S^T = KV.Q^T)"),
    (1, 64, 1, 1, "PV of a 64-head tile (O^T = V^T.P^T)"),
    (1, 64, 1, 0, "PV with P^T K-major"),
    (1, 128, 0, 0, "K-major, N = 128"),
    (1, 128, 1, 1, "MN-major, N = 128"),
    (1, 256, 0, 0, "K-major, N = 256"),
    (2, 128, 0, 0, "QK of 128 heads over a CTA pair"),
    (2, 128, 1, 1, "PV of 128 heads over a CTA pair"),
    (2, 128, 1, 0, "pair PV with P^T K-major"),
    (2, 256, 0, 0, "K-major, N = 256, pair"),
    (2, 256, 1, 1, "MN-major, N = 256, pair"),
]

# (N, A MN-major, B MN-major, chains): cta_group::1 MMAs that take 2 or 4
# accumulators in turn, against one chain of the same shape above
CHAIN_SHAPES = [
    (16, 0, 0, 2), (16, 0, 0, 4), (32, 0, 0, 2), (32, 0, 0, 4), (64, 0, 0, 2), (64, 0, 0, 4),
    (64, 1, 1, 2), (64, 1, 1, 4), (128, 0, 0, 2),
]


def _lib():
    from sparse_mla_decode_gb300 import build

    build.build()
    lib = ctypes.CDLL(build.PEAK_LIBRARY)
    lib.smla_peak_mma.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_longlong),
                                                       ctypes.POINTER(ctypes.c_float)]
    lib.smla_peak_mma.restype = ctypes.c_int
    lib.smla_peak_mma_chains.argtypes = [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_longlong),
                                                              ctypes.POINTER(ctypes.c_float)]
    lib.smla_peak_mma_chains.restype = ctypes.c_int
    lib.smla_peak_mma_commit4.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_longlong),
                                                               ctypes.POINTER(ctypes.c_float)]
    lib.smla_peak_mma_commit4.restype = ctypes.c_int
    lib.smla_peak_mma_contend.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_longlong)]
    lib.smla_peak_mma_contend.restype = ctypes.c_int
    return lib


def measure(sms: int, iters_one: int = 1000, iters_all: int = 4000):
    lib = _lib()
    rows = []
    for cg, n, amn, bmn, use in SHAPES:
        cyc = ctypes.c_longlong(0)
        ms = ctypes.c_float(0.0)
        rc = lib.smla_peak_mma(cg, n, amn, bmn, iters_one, cg, ctypes.byref(cyc), ctypes.byref(ms))
        if rc != 0:
            raise RuntimeError(f"smla_peak_mma({cg}, {n}, {amn}, {bmn}) one CTA: {rc}")
        per_mma = cyc.value / (4 * iters_one)
        ctas = (sms // cg) * cg
        rc = lib.smla_peak_mma(cg, n, amn, bmn, iters_all, ctas, ctypes.byref(cyc), ctypes.byref(ms))
        if rc != 0:
            raise RuntimeError(f"smla_peak_mma({cg}, {n}, {amn}, {bmn}) all SMs: {rc}")
        flops = ctas * 128 * n * 32 * 2 * 4 * iters_all
        rows.append({
            "cta_group": cg, "n": n, "a_mn_major": bool(amn), "b_mn_major": bool(bmn), "use": use,
            "cycles_per_mma": round(per_mma, 2), "ideal_cycles": n / 2,
            "tflops": round(flops / (ms.value * 1e-3) / 1e12, 1), "ctas": ctas,
        })
    return rows


def measure_chains(sms: int, iters_one: int = 1000, iters_all: int = 4000):
    lib = _lib()
    rows = []
    for n, amn, bmn, ch in CHAIN_SHAPES:
        cyc = ctypes.c_longlong(0)
        ms = ctypes.c_float(0.0)
        rc = lib.smla_peak_mma_chains(1, n, amn, bmn, ch, iters_one, 1, ctypes.byref(cyc), ctypes.byref(ms))
        if rc != 0:
            raise RuntimeError(f"smla_peak_mma_chains({n}, {amn}, {bmn}, {ch}) one CTA: {rc}")
        per_mma = cyc.value / (4 * iters_one)
        rc = lib.smla_peak_mma_chains(1, n, amn, bmn, ch, iters_all, sms, ctypes.byref(cyc), ctypes.byref(ms))
        if rc != 0:
            raise RuntimeError(f"smla_peak_mma_chains({n}, {amn}, {bmn}, {ch}) all SMs: {rc}")
        flops = sms * 128 * n * 32 * 2 * 4 * iters_all
        rows.append({"n": n, "a_mn_major": bool(amn), "b_mn_major": bool(bmn), "chains": ch,
                     "cycles_per_mma": round(per_mma, 2), "ideal_cycles": n / 2,
                     "tflops": round(flops / (ms.value * 1e-3) / 1e12, 1)})
    return rows


def measure_commits(sms: int, iters_one: int = 1000, iters_all: int = 4000):
    """N = 64 with a tcgen05.commit after every four MMAs."""
    lib = _lib()
    rows = []
    for mn in (0, 1):
        cyc = ctypes.c_longlong(0)
        ms = ctypes.c_float(0.0)
        rc = lib.smla_peak_mma_commit4(64, mn, mn, iters_one, 1, ctypes.byref(cyc), ctypes.byref(ms))
        if rc != 0:
            raise RuntimeError(f"smla_peak_mma_commit4({mn}) one CTA: {rc}")
        per_mma = cyc.value / (4 * iters_one)
        rc = lib.smla_peak_mma_commit4(64, mn, mn, iters_all, sms, ctypes.byref(cyc), ctypes.byref(ms))
        if rc != 0:
            raise RuntimeError(f"smla_peak_mma_commit4({mn}) all SMs: {rc}")
        flops = sms * 128 * 64 * 32 * 2 * 4 * iters_all
        rows.append({"n": 64, "a_mn_major": bool(mn), "b_mn_major": bool(mn), "commit_every": 4,
                     "cycles_per_mma": round(per_mma, 2), "tflops": round(flops / (ms.value * 1e-3) / 1e12, 1)})
    return rows


CONTEND = [(1, "three warps loading and storing 16 TMEM columns at a time"),
           (2, "a BF16 kind::f16 MMA (K = 16) before every four FP8 MMAs"),
           (3, "three warps storing 16 bytes a lane into shared memory"),
           (4, "two warps running FMA chains on the issuing warp's sub-partition"),
           (5, "nothing: the issue of the first four MMAs and their commit alone")]


def measure_contention(iters: int = 1000):
    """N = 64 K-major FP8 MMAs of one CTA beside other work."""
    lib = _lib()
    rows = []
    for mode, what in CONTEND:
        cyc = ctypes.c_longlong(0)
        rc = lib.smla_peak_mma_contend(mode, iters, ctypes.byref(cyc))
        if rc != 0:
            raise RuntimeError(f"smla_peak_mma_contend({mode}): {rc}")
        mmas = 4 if mode == 5 else iters * (5 if mode == 2 else 4)
        rows.append({"mode": mode, "beside": what, "cycles_per_mma": round(cyc.value / mmas, 2),
                     "cycles_per_fp8_mma": round(cyc.value / (4 if mode == 5 else 4 * iters), 2)})
    return rows


def clocks():
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm", "--format=csv,noheader,nounits"],
                             capture_output=True, text=True, timeout=20).stdout.strip().splitlines()[0]
        cur, mx = (float(x) for x in out.split(","))
        return {"sm_mhz_after": cur, "sm_max_mhz": mx}
    except Exception:  # noqa: BLE001 - informational only
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--json", default=None, help="write the table as JSON here")
    args = ap.parse_args()
    import torch

    props = torch.cuda.get_device_properties(0)
    rows = measure(props.multi_processor_count)
    chains = measure_chains(props.multi_processor_count)
    commits = measure_commits(props.multi_processor_count)
    contention = measure_contention()
    peak = max(r["tflops"] for r in rows)
    result = {"gpu": props.name, "sms": props.multi_processor_count, "fp8_dense_peak_tflops": peak,
              "how": "libsmla_peak.so: every SM issues 16000 tcgen05.mma kind::f8f6f4 (K = 32) into one TMEM "
                     "accumulator; FLOPs / CUDA-event time of the launch",
              "clocks": clocks(), "shapes": rows, "chains": chains, "commit_every_4": commits,
              "contention": contention}
    print("| cta_group | N | A | B | cycles/MMA | ideal | TFLOP/s (all SMs) | use |")
    print("|---|---|---|---|---|---|---|---|")
    for r in rows:
        print(f"| {r['cta_group']} | {r['n']} | {'MN' if r['a_mn_major'] else 'K'} | "
              f"{'MN' if r['b_mn_major'] else 'K'} | {r['cycles_per_mma']} | {r['ideal_cycles']:.0f} | "
              f"{r['tflops']} | {r['use']} |")
    print()
    print("| N | A | B | chains | cycles/MMA | ideal | TFLOP/s (all SMs) |")
    print("|---|---|---|---|---|---|---|")
    for r in chains:
        print(f"| {r['n']} | {'MN' if r['a_mn_major'] else 'K'} | {'MN' if r['b_mn_major'] else 'K'} | "
              f"{r['chains']} | {r['cycles_per_mma']} | {r['ideal_cycles']:.0f} | {r['tflops']} |")
    print()
    print("| N | A | B | commit every | cycles/MMA | TFLOP/s (all SMs) |")
    print("|---|---|---|---|---|---|")
    for r in commits:
        print(f"| {r['n']} | {'MN' if r['a_mn_major'] else 'K'} | {'MN' if r['b_mn_major'] else 'K'} | 4 | "
              f"{r['cycles_per_mma']} | {r['tflops']} |")
    print()
    print("| N = 64 K-major FP8 MMAs beside | cycles per MMA | cycles per FP8 MMA |")
    print("|---|---|---|")
    for r in contention:
        print(f"| {r['beside']} | {r['cycles_per_mma']} | {r['cycles_per_fp8_mma']} |")
    print(json.dumps({"fp8_dense_peak_tflops": peak}))
    if args.json:
        with open(args.json, "w") as f:
            json.dump(result, f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    sys.exit(main())
