"""Builds libsmla.so (the CUDA kernels + C ABI) in-tree for sm_103a with nvcc.

    python -m sparse_mla_decode_gb300.build [--force]

The library lands in ``sparse_mla_decode_gb300/_build/libsmla.so`` (git-ignored).
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
SOURCES = [os.path.join(CSRC, n) for n in ("smla_decode.cu", "smla_merge.cu", "smla_quant.cu", "smla_value.cu")]
HEADERS = [os.path.join(CSRC, n) for n in ("smla_ptx.cuh", "smla_merge_row.cuh")] + [os.path.join(INCLUDE, "smla.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsmla.so")


def up_to_date() -> bool:
    if not os.path.exists(LIBRARY):
        return False
    t = os.path.getmtime(LIBRARY)
    return all(os.path.getmtime(f) <= t for f in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIBRARY + f".{os.getpid()}.tmp"
    cmd = [
        nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
        "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
        "-Xlinker", "-rpath=" + os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64"),
        "-I", INCLUDE, "-o", tmp, *SOURCES,
    ]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
