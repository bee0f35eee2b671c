"""ctypes front end of the CPU oracle (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU leg may
import this module.  It compiles ``smla_oracle.c`` with gcc on first use (or
through :func:`build`) and exposes the two oracle modes over numpy arrays:

* :func:`fp64` -- the plain definition of sparse MLA decode (DeepSeek-V4.1
  ``sparse_mla_cute`` page, module docstring, "What this module computes").
* :func:`emulate` -- the Kimi K3.1 ``attn_sparse`` datapath (module docstring,
  the per-chunk softmax with E4M3 P at 448 of the running max, and
  ``SparseDcpDecode.merge``) replayed on a given (splits, chunk) partition.
* :func:`mxfp4_q_quant` -- the MXFP4 quantisation of the indexer query (Kimi
  K3.1 ``dsa_indexer_mxfp4`` page: UE8M0 scale per 32 values, E2M1 codes).
* :func:`value_gate` -- the value projection (W_UV) and sigmoid gate after
  the merge (the ``mla/dcp`` page, ``DcpValue``).
* :func:`merge` / :func:`merge_f64` -- the LSE merge of partial (out, lse) sets
  of the Kimi K3.1 ``mla/dcp`` page (``DcpValue``: weights exp2(lse - max) /
  sum, an FP32 weighted sum of the BF16 rows, one BF16 rounding).

It shares no code with the CUDA path and never imports it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "smla_oracle.c")
LIBRARY = os.path.join(HERE, "_build", "libsmla_oracle.so")

NO_P_ROUNDING = 1
EXACT = 2
P_UP = 4
P_DOWN = 8
LATENT = 512

_lock = threading.Lock()
_lib = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("width", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("num_pools", ctypes.c_int32),
        ("pool_split", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("q_stride_token", ctypes.c_int64),
        ("q_stride_head", ctypes.c_int64),
        ("pool", ctypes.c_void_p * 2),
        ("pool_rows", ctypes.c_int64 * 2),
        ("indices", ctypes.c_void_p),
        ("idx_stride_token", ctypes.c_int64),
        ("lens", ctypes.c_void_p),
        ("sinks", ctypes.c_void_p),
        ("bmm1_scale", ctypes.c_double),
        ("bmm2_scale", ctypes.c_double),
        ("k_scale", ctypes.c_double),
    ]


class _MergeProblem(ctypes.Structure):
    _fields_ = [
        ("sources", ctypes.c_int32),
        ("tokens", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("parts", ctypes.c_void_p),
        ("part_stride_source", ctypes.c_int64),
        ("part_stride_token", ctypes.c_int64),
        ("part_stride_head", ctypes.c_int64),
        ("lses", ctypes.c_void_p),
        ("lse_stride_source", ctypes.c_int64),
        ("lse_stride_token", ctypes.c_int64),
        ("lens", ctypes.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` (gcc, OpenMP, no FP contraction)."""
    if not force and os.path.exists(LIBRARY) and os.path.getmtime(LIBRARY) >= max(
        os.path.getmtime(SOURCE), os.path.getmtime(os.path.join(HERE, "smla_oracle.h"))
    ):
        return LIBRARY
    os.makedirs(os.path.dirname(LIBRARY), exist_ok=True)
    tmp = LIBRARY + f".{os.getpid()}.tmp"
    cmd = [
        "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
        "-ffp-contract=off", "-fno-fast-math", "-Wall",
        "-o", tmp, SOURCE, "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Problem)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            lib.smla_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.smla_oracle_e4m3_to_double.restype = ctypes.c_double
            lib.smla_oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.smla_oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.smla_oracle_bf16_from_float.argtypes = [ctypes.c_float]
            lib.smla_oracle_bf16_from_float.restype = ctypes.c_uint16
            lib.smla_oracle_fp64_pairs.argtypes = [P, vp, vp, i32, vp, vp, i32]
            lib.smla_oracle_emulate_pairs.argtypes = [P, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, i32]
            lib.smla_oracle_max_threads.restype = i32
            lib.smla_oracle_merge_f64.argtypes = [i32, vp, vp, vp, vp]
            lib.smla_oracle_e2m1_from_float.argtypes = [ctypes.c_float]
            lib.smla_oracle_e2m1_from_float.restype = ctypes.c_uint8
            lib.smla_oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
            lib.smla_oracle_e2m1_to_double.restype = ctypes.c_double
            lib.smla_oracle_mxfp4_q_quant.argtypes = [i32, i32, vp, vp, ctypes.c_float, vp, vp, vp]
            lib.smla_oracle_value_gate.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp]
            lib.smla_oracle_merge_pairs.argtypes = [ctypes.POINTER(_MergeProblem), vp, vp, i32, vp, vp, vp, i32]
            del i64
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().smla_oracle_max_threads())


def e4m3_to_double(byte: int) -> float:
    return float(_load().smla_oracle_e4m3_to_double(int(byte)))


def e4m3_from_float(value: float) -> int:
    return int(_load().smla_oracle_e4m3_from_float(float(value)))


def bf16_from_float(value: float) -> int:
    return int(_load().smla_oracle_bf16_from_float(float(value)))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Problem:
    """Host copy of one decode problem, held alive for the C structure.

    ``q`` uint8 [T, H, D]; ``pools`` list of uint8 [rows, D]; ``indices`` int32
    [T, W]; ``lens`` int32 [T]; ``sinks`` float32 [H] or None."""

    def __init__(self, q, pools, indices, lens, sinks, bmm1_scale, bmm2_scale, k_scale,
                 pool_split=0):
        self.q = _c(q, np.uint8)
        self.pools = [_c(p, np.uint8) for p in pools]
        self.indices = _c(indices, np.int32)
        self.lens = _c(lens, np.int32)
        self.sinks = None if sinks is None else _c(sinks, np.float32)
        T, H, D = self.q.shape
        W = self.indices.shape[1]
        s = _Problem()
        s.tokens, s.heads, s.width, s.head_dim = T, H, W, D
        s.num_pools = len(self.pools)
        s.pool_split = int(pool_split)
        s.q = self.q.ctypes.data
        s.q_stride_token, s.q_stride_head = H * D, D
        for i, p in enumerate(self.pools):
            assert p.ndim == 2 and p.shape[1] == D
            s.pool[i] = p.ctypes.data
            s.pool_rows[i] = p.shape[0]
        if len(self.pools) == 1:
            s.pool[1] = self.pools[0].ctypes.data
            s.pool_rows[1] = self.pools[0].shape[0]
        s.indices = self.indices.ctypes.data
        s.idx_stride_token = W
        s.lens = self.lens.ctypes.data
        s.sinks = None if self.sinks is None else self.sinks.ctypes.data
        s.bmm1_scale, s.bmm2_scale, s.k_scale = float(bmm1_scale), float(bmm2_scale), float(k_scale)
        self.struct = s
        self.tokens, self.heads = T, H

    @classmethod
    def from_workload(cls, w):
        return cls(w["q"], w["pools"], w["indices"], w["lens"], w["sinks"], w["bmm1_scale"],
                   w["bmm2_scale"], w["k_scale"], w.get("pool_split", 0))


def _pairs(problem, pairs):
    if pairs is None:
        t, h = np.meshgrid(np.arange(problem.tokens), np.arange(problem.heads), indexing="ij")
        return _c(t.ravel(), np.int32), _c(h.ravel(), np.int32)
    pairs = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)
    return _c(pairs[:, 0], np.int32), _c(pairs[:, 1], np.int32)


def fp64(problem: Problem, pairs=None, threads: int = 0):
    """FP64 definition. Returns (out [n, 512] float64, lse2 [n] float64) for the
    (token, head) ``pairs`` (all pairs in row-major order when None)."""
    lib = _load()
    tok, head = _pairs(problem, pairs)
    n = tok.size
    out = np.zeros((n, LATENT), np.float64)
    lse = np.zeros(n, np.float64)
    lib.smla_oracle_fp64_pairs(ctypes.byref(problem.struct), tok.ctypes.data, head.ctypes.data,
                               n, out.ctypes.data, lse.ctypes.data, threads)
    return out, lse


def emulate(problem: Problem, splits: int, chunk: int, pairs=None, flags: int = 0,
            threads: int = 0, ties: bool = False):
    """E4M3-P datapath on the given partition. Returns (value [n, 512] float64 --
    the pre-BF16 result, bf16 [n, 512] uint16 bits, lse2 [n] float64), and with
    ``ties`` a fourth array [n, 512]: the most each value moves when every P
    within a relative 2^-16 of an E4M3 rounding midpoint takes its other code
    (a rounding the FP32 datapath leaves open)."""
    lib = _load()
    tok, head = _pairs(problem, pairs)
    n = tok.size
    value = np.zeros((n, LATENT), np.float64)
    bits = np.zeros((n, LATENT), np.uint16)
    lse = np.zeros(n, np.float64)
    tie = np.zeros((n, LATENT), np.float64)
    rc = lib.smla_oracle_emulate_pairs(ctypes.byref(problem.struct), tok.ctypes.data,
                                       head.ctypes.data, n, int(splits), int(chunk), int(flags),
                                       value.ctypes.data, bits.ctypes.data, lse.ctypes.data,
                                       tie.ctypes.data, threads)
    if rc != 0:
        raise ValueError("oracle emulate: bad partition")
    if ties:
        return value, bits, lse, tie
    return value, bits, lse


def merge_f64(rows, lses):
    """The merge in double of ``rows`` [S, 512] with base-2 ``lses`` [S].
    Returns (out [512] float64, lse2 float)."""
    lib = _load()
    rows = _c(rows, np.float64).reshape(-1, LATENT)
    lses = _c(lses, np.float64).reshape(-1)
    assert rows.shape[0] == lses.size
    out = np.zeros(LATENT, np.float64)
    lse = np.zeros(1, np.float64)
    lib.smla_oracle_merge_f64(int(lses.size), rows.ctypes.data, lses.ctypes.data, out.ctypes.data,
                              lse.ctypes.data)
    return out, float(lse[0])


class MergeProblem:
    """Host copy of one merge problem: ``parts`` BF16 bits uint16 [S, T, H, 512],
    ``lses`` float32 [S, T, H] (base 2), ``lens`` int32 [T] or None."""

    def __init__(self, parts, lses, lens=None):
        self.parts = _c(parts, np.uint16)
        self.lses = _c(lses, np.float32)
        self.lens = None if lens is None else _c(lens, np.int32)
        S, T, H, J = self.parts.shape
        assert J == LATENT and self.lses.shape == (S, T, H)
        m = _MergeProblem()
        m.sources, m.tokens, m.heads = S, T, H
        m.parts = self.parts.ctypes.data
        m.part_stride_source, m.part_stride_token, m.part_stride_head = T * H * J, H * J, J
        m.lses = self.lses.ctypes.data
        m.lse_stride_source, m.lse_stride_token = T * H, H
        m.lens = None if self.lens is None else self.lens.ctypes.data
        self.struct = m
        self.tokens, self.heads = T, H


def merge(problem: MergeProblem, pairs=None, threads: int = 0):
    """LSE merge of the (token, head) ``pairs`` (all, row-major, when None).
    Returns (value [n, 512] float64 before rounding, bf16 [n, 512] uint16 bits,
    lse2 [n] float64)."""
    lib = _load()
    tok, head = _pairs(problem, pairs)
    n = tok.size
    value = np.zeros((n, LATENT), np.float64)
    bits = np.zeros((n, LATENT), np.uint16)
    lse = np.zeros(n, np.float64)
    rc = lib.smla_oracle_merge_pairs(ctypes.byref(problem.struct), tok.ctypes.data, head.ctypes.data, n,
                                     value.ctypes.data, bits.ctypes.data, lse.ctypes.data, threads)
    if rc != 0:
        raise MemoryError("oracle merge")
    return value, bits, lse


def e2m1_from_float(value: float) -> int:
    return int(_load().smla_oracle_e2m1_from_float(float(value)))


def e2m1_to_double(code: int) -> float:
    return float(_load().smla_oracle_e2m1_to_double(int(code)))


def mxfp4_q_quant(q, weights, weight_scale: float, padded_heads: int):
    """MXFP4 of the indexer query ``q`` float32 [T, H, 128] (values as FP32)
    and the scaled ``weights`` float32 [T, H]. Returns (packed uint8 [T, P, 64],
    scale int32 [T, P], weights float32 [T, P])."""
    lib = _load()
    q = _c(q, np.float32)
    weights = _c(weights, np.float32)
    T, H, D = q.shape
    assert D == 128 and weights.shape == (T, H) and padded_heads >= H
    P = int(padded_heads)
    packed = np.zeros((T, P, 64), np.uint8)
    scale = np.zeros((T, P), np.int32)
    w_out = np.zeros((T, P), np.float32)
    for t in range(T):
        lib.smla_oracle_mxfp4_q_quant(H, P, q[t].ctypes.data, weights[t].ctypes.data, float(weight_scale),
                                      packed[t].ctypes.data, scale[t].ctypes.data, w_out[t].ctypes.data)
    return packed, scale, w_out


def value_gate(latent_bits, w_bits, gate_bits, lens=None):
    """out[t, h*128 + v] = BF16(BF16(sum_j latent[t,h,j] W[h,j,v]) * sigmoid(gate[t, h*128+v])).
    latent_bits uint16 [T, H, 512], w_bits uint16 [H, 512, 128], gate_bits
    uint16 [T, H*128]; returns (value [T, H*128] float64, bits uint16)."""
    lib = _load()
    latent = _c(latent_bits, np.uint16)
    w = _c(w_bits, np.uint16)
    gate = _c(gate_bits, np.uint16)
    T, H, J = latent.shape
    assert J == LATENT and w.shape == (H, LATENT, 128) and gate.shape == (T, H * 128)
    lens = None if lens is None else _c(lens, np.int32)
    value = np.zeros((T, H * 128), np.float64)
    bits = np.zeros((T, H * 128), np.uint16)
    lib.smla_oracle_value_gate(T, H, latent.ctypes.data, w.ctypes.data, gate.ctypes.data,
                               None if lens is None else lens.ctypes.data, value.ctypes.data, bits.ctypes.data)
    return value, bits
