"""Pins of the fp8_ds_mla oracle (``oracle/ds_mla.py``) to facts outside it.

* The dequantisation against torch's E4M3 and BF16 decoders (library routines).
* A reduction to the 576-byte decode oracle (DeepSeek-V4.1 ``sparse_mla_cute``
  page, "What this module computes"): rows whose scales are 1 and whose rope
  values are the E4M3 rope values give that oracle's result with
  ``k_scale = 1``.
* A per-block scale-transfer invariant: moving a power of two from Q's latent
  block b into the scale of block b leaves the logits unchanged and scales
  output block b by it. A wrong block index (``j % 4`` for ``j // 128``) or a
  scale on the rope breaks it.
* The single-key case: the output is bmm2_scale times the dequantised row.
"""

import math

import numpy as np
import pytest
import torch

from oracle import ds_mla, oracle


def random_rows(rng, R):
    codes = torch.from_numpy(rng.standard_normal((R, 512)).astype(np.float32)).to(torch.float8_e4m3fn)
    codes = codes.view(torch.uint8).numpy()
    scales = (2.0 ** rng.integers(-6, 3, (R, 4)) * rng.uniform(0.5, 1.0, (R, 4))).astype(np.float32)
    rope = torch.from_numpy(rng.standard_normal((R, 64)).astype(np.float32)).to(torch.bfloat16)
    rope_bits = rope.view(torch.int16).numpy().view(np.uint16)
    return ds_mla.encode_rows(codes, scales, rope_bits), codes, scales, rope


def test_dequantisation_matches_the_library_decoders():
    rng = np.random.default_rng(1)
    rows, codes, scales, rope = random_rows(rng, 7)
    got = ds_mla.dequant_rows(rows)
    lat = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    want_lat = lat * np.repeat(scales.astype(np.float64), 128, axis=1)
    np.testing.assert_array_equal(got[:, :512], want_lat)
    np.testing.assert_array_equal(got[:, 512:], rope.to(torch.float64).numpy())


def test_reduces_to_the_576_byte_definition():
    """576-byte E4M3 rows against the same values as fp8_ds_mla rows: scales 1,
    rope values exactly the E4M3 ones (E4M3 values are exact in BF16)."""
    rng = np.random.default_rng(2)
    T, H, W, R = 3, 4, 40, 300
    pool576 = torch.from_numpy(rng.standard_normal((R, 576)).astype(np.float32)).to(torch.float8_e4m3fn)
    pool576 = pool576.view(torch.uint8).numpy()
    q576 = torch.from_numpy(rng.standard_normal((T, H, 576)).astype(np.float32)).to(torch.float8_e4m3fn)
    q576 = q576.view(torch.uint8).numpy()
    indices = rng.choice(R, (T, W)).astype(np.int32)
    indices[rng.random((T, W)) < 0.1] = -1
    lens = np.array([W, 17, 0], np.int32)
    sinks = rng.standard_normal(H).astype(np.float32)
    bmm1, bmm2 = 1.0 / math.sqrt(192.0), 0.75
    ref, ref_lse = oracle.fp64(oracle.Problem(q576, [pool576], indices, lens, sinks, bmm1, bmm2, 1.0))

    rope_vals = torch.from_numpy(pool576[:, 512:].copy()).view(torch.float8_e4m3fn).to(torch.bfloat16)
    rows = ds_mla.encode_rows(pool576[:, :512], np.ones((R, 4), np.float32),
                              rope_vals.view(torch.int16).numpy().view(np.uint16))
    qv = torch.from_numpy(q576).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    out, lse = ds_mla.fp64(qv, rows, indices, lens, sinks.astype(np.float64), bmm1, bmm2)
    np.testing.assert_allclose(out.reshape(T * H, 512), ref, rtol=1e-12, atol=1e-14)
    assert np.all(np.isneginf(lse[2])) and np.all(out[2] == 0.0)
    np.testing.assert_allclose(lse.reshape(-1)[:2 * H], ref_lse[:2 * H], rtol=1e-12)


@pytest.mark.parametrize("block", [0, 1, 2, 3])
def test_scale_moved_from_q_to_a_block_scales_that_output_block(block):
    rng = np.random.default_rng(3 + block)
    T, H, W, R = 2, 3, 24, 64
    rows, codes, scales, rope = random_rows(rng, R)
    q = rng.standard_normal((T, H, 576))
    indices = rng.choice(R, (T, W), replace=False).astype(np.int32)
    lens = np.array([W, 9], np.int32)
    out, lse = ds_mla.fp64(q, rows, indices, lens, None, 0.1, 1.0)

    c = 4.0  # a power of two: the FP32 scales and the logits stay exact
    scales2 = scales.copy()
    scales2[:, block] *= c
    rope_bits = rows[:, 528:].copy().view("<u2")
    rows2 = ds_mla.encode_rows(codes, scales2, rope_bits)
    q2 = q.copy()
    q2[:, :, 128 * block:128 * (block + 1)] /= c
    out2, lse2 = ds_mla.fp64(q2, rows2, indices, lens, None, 0.1, 1.0)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12)
    want = out.copy()
    want[:, :, 128 * block:128 * (block + 1)] *= c
    np.testing.assert_allclose(out2, want, rtol=1e-12, atol=1e-15)


def test_single_active_key_returns_the_scaled_row():
    rng = np.random.default_rng(9)
    rows, _, _, _ = random_rows(rng, 5)
    q = rng.standard_normal((1, 2, 576))
    indices = np.array([[3, -1, 7]], np.int32)  # 7 is past the pool: a hole
    out, lse = ds_mla.fp64(q, rows, indices, np.array([3], np.int32), None, 0.2, 0.5)
    row = ds_mla.dequant_rows(rows[3:4])[0]
    np.testing.assert_allclose(out[0], 0.5 * np.tile(row[:512], (2, 1)), rtol=1e-14)
    np.testing.assert_allclose(lse[0], 0.2 * (q[0] @ row) / math.log(2.0), rtol=1e-12)
