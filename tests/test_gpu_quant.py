"""GPU parity of the MXFP4 indexer-query quantisation (``smla_mxfp4_q_quant``)
against the oracle (the Kimi K3.1 dsa_indexer_mxfp4 page): the packed E2M1
codes, the UE8M0 scale bytes and the scaled weights are integer or exact
results, so they must match bit for bit."""

import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_mla_decode_gb300 import smla

pytestmark = pytest.mark.gpu


def inputs(seed, T, H, dtype):
    """Normal values with a per-head magnitude over 12 decades, plus edge
    blocks: all zero, all negative zero, amax exactly 6 * 2^k and one ulp
    above, tiny and huge magnitudes, and values on the E2M1 midpoints."""
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((T, H, 128)) * 10.0 ** rng.uniform(-6, 6, (T, H, 1))).astype(np.float32)
    if T >= 1 and H >= 4:
        q[0, 0, 0:32] = 0.0
        q[0, 0, 32:64] = -0.0
        q[0, 1, 0:32] = 6.0 * 2.0 ** 5
        q[0, 1, 32:64] = np.nextafter(np.float32(6.0 * 2.0 ** -7), np.float32(1.0))
        q[0, 2, 0:32] = np.float32(1e-39)  # subnormal
        q[0, 2, 32:64] = np.float32(3e38)
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -1.75, -5.0], np.float32)
        q[0, 3, 0:32] = np.resize(mids, 32)
        q[0, 3, 0] = 6.0  # keeps the block scale at 2^0 so the midpoints stay midpoints
    w = rng.standard_normal((T, H)).astype(np.float32)
    qt = torch.from_numpy(q)
    if dtype == torch.bfloat16:
        qt = qt.to(torch.bfloat16)
        q = qt.float().numpy()  # the values the kernel sees
    return qt, q, w


def check(qt, q, w, scale, P):
    packed, sc, wo = smla.mxfp4_q_quant(qt.cuda(), torch.from_numpy(w).cuda(), scale, padded_heads=P)
    torch.cuda.synchronize()
    ref_packed, ref_scale, ref_w = oracle.mxfp4_q_quant(q, w, scale, P)
    got_packed = packed.cpu().numpy()
    diff = np.argwhere(got_packed != ref_packed)
    assert diff.size == 0, f"{len(diff)} packed bytes differ, first at {diff[:3]}: " \
                           f"{got_packed[tuple(diff[0])]:#x} vs {ref_packed[tuple(diff[0])]:#x}"
    assert np.array_equal(sc.cpu().numpy(), ref_scale)
    assert np.array_equal(wo.cpu().numpy().view(np.uint32), ref_w.view(np.uint32))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("T,H,P", [(1, 4, 4), (3, 32, 32), (5, 20, 32), (64, 64, 64)])
def test_mxfp4_matches_the_oracle_bit_for_bit(dtype, T, H, P):
    qt, q, w = inputs(T * 100 + H, T, H, dtype)
    check(qt, q, w, 0.0625, P)


def test_mxfp4_strided_query():
    qt, q, w = inputs(55, 4, 8, torch.float32)
    big = torch.zeros((4, 10, 136), dtype=torch.float32)
    big[:, :8, :128] = qt
    packed, sc, wo = smla.mxfp4_q_quant(big.cuda()[:, :8, :128], torch.from_numpy(w).cuda(), 0.5, padded_heads=8)
    ref, ref_sc, ref_w = smla.mxfp4_q_quant(qt.cuda(), torch.from_numpy(w).cuda(), 0.5, padded_heads=8)
    torch.cuda.synchronize()
    assert torch.equal(packed, ref) and torch.equal(sc, ref_sc) and torch.equal(wo, ref_w)


def test_mxfp4_no_tokens_is_a_no_op():
    q = torch.empty((0, 32, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.empty((0, 32), dtype=torch.float32, device="cuda")
    packed, sc, wo = smla.mxfp4_q_quant(q, w, 1.0, padded_heads=64)
    assert packed.shape == (0, 64, 64)


def test_mxfp4_prefill_size_sampled():
    """16384 tokens x 32 heads (the pages' prefill size for this op); every
    97th token checked bit for bit."""
    T, H = 16384, 32
    gen = torch.Generator(device="cuda")
    gen.manual_seed(31)
    qt = torch.randn((T, H, 128), generator=gen, device="cuda").to(torch.bfloat16)
    w = torch.randn((T, H), generator=gen, device="cuda")
    packed, sc, wo = smla.mxfp4_q_quant(qt, w, 0.25, padded_heads=H)
    torch.cuda.synchronize()
    rows = np.arange(0, T, 97)
    q = qt[rows].float().cpu().numpy()
    ref_packed, ref_scale, ref_w = oracle.mxfp4_q_quant(q, w[rows].cpu().numpy(), 0.25, H)
    assert np.array_equal(packed[rows].cpu().numpy(), ref_packed)
    assert np.array_equal(sc[rows].cpu().numpy(), ref_scale)
    assert np.array_equal(wo[rows].cpu().numpy().view(np.uint32), ref_w.view(np.uint32))
