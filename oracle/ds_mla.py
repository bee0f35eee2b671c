"""FP64 definition of sparse MLA decode over fp8_ds_mla rows (test
infrastructure: only ``tests/`` may import this module; it shares no code with
the CUDA path).

The Kimi K3.1 ``dsa_fused_prologue`` page (the ``mla_cache`` argument and the
insert of ``[kv_c_normed | k_pe]``) gives an MLA cache row of 656 bytes and views
the cache as FP8, as float32 and as BF16. It does not print the row's layout.
The plainest reading of 656 = 512 + 16 + 128, taken here:

* R1. Bytes [0, 512) are the E4M3 codes of the 512 latents. Bytes [512, 528)
  are four little-endian FP32 scales s_0..s_3. Bytes [528, 656) are the 64 rope
  values as little-endian BF16.
* R2. Latent j dequantises to ``dec(code_j) * s_(j // 128)``: one scale per 128
  latents, the count the 16 bytes leave room for. A rope value is its BF16 value.
* R3. The attention is the 576-byte decode's definition (DeepSeek-V4.1
  ``sparse_mla_cute`` page, "What this module computes"), with K the 576
  dequantised values and V the 512 latents. The row's scales take the place of
  ``k_scale``, so the output multiplier is ``bmm2_scale`` alone. Q is given as
  values; how a kernel encodes it is the kernel's choice.

The layout reading R1 cannot be pinned against the pages (they print no row),
so the parity of R1 itself is unpinned. R2 and R3 are pinned in
``tests/test_oracle_ds_mla.py``:
* a reduction to the 576-byte definition;
* a per-block scale-transfer invariant;
* the library E4M3/BF16 decoders;
* the single-key case.
"""

from __future__ import annotations

import math

import numpy as np

from . import oracle as _oracle

ROW_BYTES = 656
LATENT = 512
ROPE = 64
SCALE_BLOCK = 128


def _e4m3_table() -> np.ndarray:
    return np.array([_oracle.e4m3_to_double(b) for b in range(256)], np.float64)


_TABLE = None


def dequant_rows(rows) -> np.ndarray:
    """uint8 [R, 656] rows (R1) -> float64 [R, 576] values (R2): 512 latents
    then 64 rope values."""
    global _TABLE
    if _TABLE is None:
        _TABLE = _e4m3_table()
    rows = np.ascontiguousarray(rows, np.uint8)
    assert rows.ndim == 2 and rows.shape[1] == ROW_BYTES
    codes = _TABLE[rows[:, :LATENT]]
    scales = rows[:, LATENT:LATENT + 16].copy().view("<f4").astype(np.float64)  # [R, 4]
    latent = codes * np.repeat(scales, SCALE_BLOCK, axis=1)
    rope_bits = rows[:, LATENT + 16:].copy().view("<u2").astype(np.uint32) << 16
    rope = rope_bits.view(np.float32).astype(np.float64)
    return np.concatenate([latent, rope], axis=1)


def fp64(q, pool, indices, lens, sinks, bmm1_scale: float, bmm2_scale: float):
    """The definition over one pool of fp8_ds_mla rows.

    q float64 [T, H, 576] values; pool uint8 [rows, 656]; indices int32 [T, W]
    (-1 = hole); lens int32 [T] (clamped to [0, W]); sinks float [H] in score
    units, or None. Returns (out float64 [T, H, 512], lse2 float64 [T, H],
    base 2). A token with no active column gets zeros and -inf, whatever its
    sink. An index at or beyond the pool's rows is a hole."""
    q = np.asarray(q, np.float64)
    T, H, D = q.shape
    assert D == LATENT + ROPE
    indices = np.asarray(indices, np.int64)
    W = indices.shape[1]
    rows = np.asarray(pool).shape[0]
    out = np.zeros((T, H, LATENT), np.float64)
    lse2 = np.full((T, H), -np.inf)
    for t in range(T):
        n = min(max(int(lens[t]), 0), W)
        cols = indices[t, :n]
        active = cols[(cols >= 0) & (cols < rows)]
        if active.size == 0:
            continue
        kv = dequant_rows(np.asarray(pool)[active])          # [A, 576]
        s = bmm1_scale * (q[t] @ kv.T)                       # [H, A]
        m = s.max(axis=1)
        if sinks is not None:
            m = np.maximum(m, np.asarray(sinks, np.float64))
        p = np.exp(s - m[:, None])
        den = p.sum(axis=1)
        if sinks is not None:
            den = den + np.exp(np.asarray(sinks, np.float64) - m)
        out[t] = bmm2_scale * (p @ kv[:, :LATENT]) / den[:, None]
        lse2[t] = (m + np.log(den)) / math.log(2.0)
    return out, lse2


def encode_rows(codes, scales, rope_bits) -> np.ndarray:
    """Assemble rows per R1 from uint8 codes [R, 512], float32 scales [R, 4]
    and uint16 BF16 rope bits [R, 64]."""
    codes = np.ascontiguousarray(codes, np.uint8)
    R = codes.shape[0]
    rows = np.zeros((R, ROW_BYTES), np.uint8)
    rows[:, :LATENT] = codes
    rows[:, LATENT:LATENT + 16] = np.ascontiguousarray(scales, "<f4").view(np.uint8).reshape(R, 16)
    rows[:, LATENT + 16:] = np.ascontiguousarray(rope_bits, "<u2").view(np.uint8).reshape(R, 2 * ROPE)
    return rows
