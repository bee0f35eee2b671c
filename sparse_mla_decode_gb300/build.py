"""Builds libsmla.so (the CUDA kernels + C ABI) in-tree for sm_103a with nvcc.

    python -m sparse_mla_decode_gb300.build [--force]

The library lands in ``sparse_mla_decode_gb300/_build/libsmla.so`` (git-ignored), beside
``libsmla_peak.so``, the FP8 tensor-core microbenchmark.
It links the CUDA runtime dynamically, so a process that already loaded
PyTorch's runtime shares it.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "libsmla.so")
PEAK_LIBRARY = os.path.join(BUILD_DIR, "libsmla_peak.so")
SOURCES = [os.path.join(CSRC, n) for n in ("smla_decode.cu", "smla_pair.cu", "smla_ds_mla.cu", "smla_merge.cu", "smla_quant.cu",
                                          "smla_value.cu")]
HEADERS = [os.path.join(CSRC, n) for n in ("smla_ptx.cuh", "smla_merge_row.cuh", "smla_pair.cuh")] + [os.path.join(INCLUDE, "smla.h")]
# the FP8 tensor-core microbenchmark, a library of its own
PEAK_SOURCES = [os.path.join(CSRC, "smla_peak.cu"), os.path.join(CSRC, "smla_peak_gather.cu")]
TARGETS = {LIBRARY: (SOURCES, HEADERS), PEAK_LIBRARY: (PEAK_SOURCES, [os.path.join(CSRC, "smla_ptx.cuh")])}
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsmla.so")


def _fresh(library: str) -> bool:
    if not os.path.exists(library):
        return False
    t = os.path.getmtime(library)
    sources, headers = TARGETS[library]
    return all(os.path.getmtime(f) <= t for f in sources + headers)


def up_to_date() -> bool:
    return all(_fresh(lib) for lib in TARGETS)


def _command(library: str, tmp: str, verbose: bool):
    cmd = [
        nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
        "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
        "-Xlinker", "-rpath=" + os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64"),
        "-I", INCLUDE, "-o", tmp, *TARGETS[library][0],
    ]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles every stale library (in parallel) and returns libsmla.so's path."""
    todo = [lib for lib in TARGETS if force or not _fresh(lib)]
    if not todo:
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    jobs = []
    for lib in todo:
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = _command(lib, tmp, verbose)
        jobs.append((lib, tmp, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                                      text=True)))
    failed = []
    for lib, tmp, cmd, proc in jobs:
        out, err = proc.communicate()
        if proc.returncode != 0:
            failed.append("nvcc failed:\n" + " ".join(cmd) + "\n" + out + err)
            continue
        if verbose:
            sys.stderr.write(err)
        os.replace(tmp, lib)
    if failed:
        raise RuntimeError("\n".join(failed))
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
