"""Random-row gather rates of this GPU: 576-byte rows at random row numbers
into shared memory, measured with the library's own microbenchmark
(``libsmla_peak.so``, built from ``csrc/smla_peak_gather.cu``).

    python -m sparse_mla_decode_gb300.gather_peak [--json PATH]

Every CTA (one per SM) streams 16 chunks of 128 rows (2048 rows, what one
CTA of the 64 x 128 x 2048 batch gathers) into a three-stage ring that
nothing consumes, by each of the ways the decode can gather: cp.async from 7
or 16 warps, TMA tile::gather4 from 1 to 16 issuing warps, and tile::gather4
with multicast in CTA pairs that share each chunk (the decode's paired head
groups; a stage is refilled once both CTAs have seen it land). Two pools:

* cold: 1,048,576 rows (604 MB), row numbers uniform per CTA (per pair for
  the multicast method), the L2 flushed (a 256 MB write) before the launch;
* hot: 32,768 rows (18.9 MB) that the L2 holds, warmed by the same launch
  first.

Per row: ``landed_gbs`` = rows x 576 bytes that reached shared memory, over
all CTAs, / the launch's CUDA-event time (median of 3); ``sm_bytes_per_ns`` =
the same per CTA; ``unique_gbs`` = distinct bytes read from the pool (half of
the landed bytes for the multicast pairs). With ``--json`` the table is
written as JSON (the summary committed under ``profiles/``).
"""

from __future__ import annotations

import argparse
import ctypes
import json
import statistics
import sys

ROW_BYTES = 576
CHUNKS = 16
ROWS_PER_CHUNK = 128
COLD_ROWS = 1 << 20
HOT_ROWS = 1 << 15

# (method, issuing warps, what it is)
METHODS = [
    (0, 7, "cp.async, 7 warps (the decode's unpaired producers)"),
    (0, 16, "cp.async, 16 warps"),
    (1, 1, "tile::gather4, 1 issuing warp"),
    (1, 4, "tile::gather4, 4 issuing warps"),
    (1, 7, "tile::gather4, 7 issuing warps"),
    (1, 16, "tile::gather4, 16 issuing warps"),
    (2, 7, "tile::gather4 multicast in CTA pairs, 7 warps (the decode's paired producers)"),
    (2, 16, "tile::gather4 multicast in CTA pairs, 16 warps"),
]


def _lib():
    from sparse_mla_decode_gb300 import build

    build.build()
    lib = ctypes.CDLL(build.PEAK_LIBRARY)
    lib.smla_peak_gather.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)]
    lib.smla_peak_gather.restype = ctypes.c_int
    return lib


def measure(sms: int, reps: int = 3):
    import torch

    lib = _lib()
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(2024)
    cold = torch.randint(0, 256, (COLD_ROWS, ROW_BYTES), dtype=torch.uint8, device=dev, generator=gen)
    hot = cold[:HOT_ROWS]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    error = torch.zeros(1, dtype=torch.int32, device=dev)
    ctas = sms - sms % 2

    def launch(method, issuers, pool, idx):
        ms = ctypes.c_float(0.0)
        rc = lib.smla_peak_gather(method, issuers, pool.data_ptr(), pool.shape[0], idx.data_ptr(), ctas, CHUNKS,
                                  error.data_ptr(), ctypes.byref(ms))
        if rc != 0 or int(error.item()) != 0:
            raise RuntimeError(f"smla_peak_gather({method}, {issuers}): rc {rc}, error {int(error.item())}")
        return ms.value

    rows_out = []
    for method, issuers, what in METHODS:
        units = ctas // 2 if method == 2 else ctas
        for kind, pool in (("cold", cold), ("hot", hot)):
            times = []
            for _ in range(reps):
                idx = torch.randint(0, pool.shape[0], (units, CHUNKS, ROWS_PER_CHUNK), dtype=torch.int32,
                                    device=dev, generator=gen)
                if kind == "cold":
                    flush.fill_(1)
                else:
                    launch(method, issuers, pool, idx)  # the rows into L2
                torch.cuda.synchronize()
                times.append(launch(method, issuers, pool, idx))
            ms = statistics.median(times)
            landed = ctas * CHUNKS * ROWS_PER_CHUNK * ROW_BYTES
            unique = landed // 2 if method == 2 else landed
            rows_out.append({
                "method": method, "issuers": issuers, "what": what, "pool": kind, "ctas": ctas,
                "us": round(ms * 1e3, 2), "landed_gbs": round(landed / (ms * 1e-3) / 1e9, 1),
                "unique_gbs": round(unique / (ms * 1e-3) / 1e9, 1),
                "sm_bytes_per_ns": round(landed / ctas / (ms * 1e6), 2),
            })
    return rows_out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--json", default=None, help="write the table as JSON here")
    args = ap.parse_args()
    import torch

    props = torch.cuda.get_device_properties(0)
    rows = measure(props.multi_processor_count)
    print("| method | pool | us | landed GB/s | unique GB/s | B/ns per SM |")
    print("|---|---|---|---|---|---|")
    for r in rows:
        print(f"| {r['what']} | {r['pool']} | {r['us']} | {r['landed_gbs']} | {r['unique_gbs']} | "
              f"{r['sm_bytes_per_ns']} |")
    best = {k: max((r for r in rows if r["pool"] == k), key=lambda r: r["unique_gbs"]) for k in ("cold", "hot")}
    summary = {k: {"unique_gbs": v["unique_gbs"], "what": v["what"]} for k, v in best.items()}
    print(json.dumps(summary))
    if args.json:
        with open(args.json, "w") as f:
            json.dump({"gpu": props.name, "sms": props.multi_processor_count, "rows_per_cta": CHUNKS * ROWS_PER_CHUNK,
                       "row_bytes": ROW_BYTES, "best": summary, "rows": rows}, f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    sys.exit(main())
