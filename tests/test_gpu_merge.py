"""GPU parity of the LSE merge of partial (out, lse) sets (``smla_merge``)
against the oracle's merge (the Kimi K3.1 mla/dcp page, DcpValue), and of
decode-then-merge against the decode definition of the whole problem."""

import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_mla_decode_gb300 import smla, workloads
from tests.gpu_helpers import TOL_FP64, bf16_ulp, e4m3_p_bound

pytestmark = pytest.mark.gpu


def random_sets(seed, S, T, H, invalid=0.1, lens_zero=()):
    """BF16 partial rows N(0, 1) and base-2 LSEs U(-6, 6) with a fraction of
    empty sources (-inf, +inf or NaN LSE); lens with the given zero tokens."""
    rng = np.random.default_rng(seed)
    parts = torch.from_numpy(rng.standard_normal((S, T, H, 512)).astype(np.float32)).to(torch.bfloat16)
    lses = rng.uniform(-6.0, 6.0, (S, T, H)).astype(np.float32)
    kinds = rng.random((S, T, H))
    lses[kinds < invalid] = -np.inf
    lses[(kinds >= invalid) & (kinds < invalid * 1.3)] = np.nan
    lses[(kinds >= invalid * 1.3) & (kinds < invalid * 1.5)] = np.inf
    lens = np.full(T, 7, np.int32)
    for t in lens_zero:
        lens[t] = 0
    return parts, lses, lens


def check(parts, lses, lens, got, got_lse):
    """Element-wise: |gpu - exact| <= 1 BF16 ulp of the exact value + 1e-6 of
    the largest source magnitude (FP32 accumulation and ex2 weights); empty
    rows +0.0 / -inf bit-exact; |lse - exact| <= 1e-5 (1 + |exact|)."""
    bits = parts.view(torch.int16).numpy().view(np.uint16)
    value, ref_bits, ref_lse = oracle.merge(oracle.MergeProblem(bits, lses, lens))
    g = got.float().cpu().numpy().reshape(value.shape)
    gb = got.view(torch.int16).cpu().numpy().view(np.uint16).reshape(value.shape)
    gl = got_lse.cpu().numpy().reshape(-1)
    empty = np.isneginf(ref_lse)
    assert np.all(gb[empty] == 0), "empty rows must be +0.0"
    assert np.all(np.isneginf(gl[empty])), "empty rows must have LSE -inf"
    live = ~empty
    if live.any():
        scale = np.abs(parts.float().numpy()).reshape(parts.shape[0], -1, 512).max(axis=(0, 2))[live]
        err = np.abs(g[live] - value[live])
        bound = bf16_ulp(value[live]) + 1e-6 * scale[:, None]
        worst = float((err / bound).max())
        assert worst <= 1.0, f"merge error at {worst:.3f} of the bound"
        lerr = np.abs(gl[live] - ref_lse[live]) / (1.0 + np.abs(ref_lse[live]))
        assert lerr.max() <= 1e-5, f"merged LSE error {lerr.max()}"
        same = float(np.mean(gb[live] == ref_bits[live]))
        print(f"merge: worst {worst:.3f} of the bound, {same:.5f} of the bits equal")


@pytest.mark.parametrize("S,T,H", [(1, 3, 16), (2, 2, 32), (3, 5, 16), (5, 4, 64), (8, 3, 128), (37, 2, 16), (70, 3, 16)])
def test_merge_matches_the_oracle(S, T, H):
    """Up to 64 sources a warp loads its next row's LSEs ahead; beyond, the
    kernel takes each row's LSEs with it (70 here)."""
    parts, lses, lens = random_sets(100 + S, S, T, H, lens_zero=(1,) if T > 2 else ())
    d = parts.cuda()
    out, lse = smla.merge(d, torch.from_numpy(lses).cuda(), torch.from_numpy(lens).cuda())
    torch.cuda.synchronize()
    check(parts, lses, lens, out, lse)


def test_merge_of_no_sources_is_empty():
    out = torch.full((2, 16, 512), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((2, 16), dtype=torch.float32, device="cuda")
    parts = torch.empty((0, 2, 16, 512), dtype=torch.bfloat16, device="cuda")
    lses = torch.empty((0, 2, 16), dtype=torch.float32, device="cuda")
    smla.smla_merge(parts, lses, None, out, lse)
    torch.cuda.synchronize()
    assert torch.all(out.view(torch.int16) == 0) and torch.all(torch.isneginf(lse))


def test_merge_strided_layouts_match_contiguous():
    parts, lses, lens = random_sets(7, 4, 3, 32)
    d = parts.cuda()
    ref_out, ref_lse = smla.merge(d, torch.from_numpy(lses).cuda(), torch.from_numpy(lens).cuda())
    # sources interleaved per token ([T, S, H, 512] storage), heads padded, out inside a wider buffer
    big = torch.zeros((3, 4, 40, 520), dtype=torch.bfloat16, device="cuda")
    big[:, :, :32, :512] = d.permute(1, 0, 2, 3)
    sparts = big[:, :, :32, :512].permute(1, 0, 2, 3)
    lbig = torch.zeros((3, 4, 48), dtype=torch.float32, device="cuda")
    lbig[:, :, :32] = torch.from_numpy(lses).cuda().permute(1, 0, 2)
    slses = lbig[:, :, :32].permute(1, 0, 2)
    obig = torch.zeros((3, 36, 528), dtype=torch.bfloat16, device="cuda")
    out = obig[:, :32, :512]
    lbuf = torch.zeros((3, 40), dtype=torch.float32, device="cuda")
    smla.smla_merge(sparts, slses, torch.from_numpy(lens).cuda(), out, lbuf[:, :32])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lbuf[:, :32], ref_lse)


def test_decode_shards_then_merge_equal_the_whole_decode():
    """Split every token's columns into 3 key shards, decode each shard with
    smla_decode (BF16 rows + base-2 LSEs), merge the shards with smla_merge, and
    compare with the fp64 decode of all columns (the decode tolerance, plus one
    BF16 rounding per shard)."""
    w = workloads.small("shards", seed=303, tokens=3, heads=64, width=900, head_dim=576, pool_rows=5000,
                        holes=0.05, lens=[900, 500, 33])
    W = w["indices"].shape[1]
    bounds = [0, 300, 620, W]
    outs, lses = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        sub = dict(w)
        sub["indices"] = np.full_like(w["indices"], -1)
        sub["indices"][:, a:b] = w["indices"][:, a:b]
        q = torch.from_numpy(sub["q"]).cuda()
        o, l = smla.decode(q, [torch.from_numpy(p).cuda() for p in sub["pools"]],
                           torch.from_numpy(sub["indices"]).cuda(), torch.from_numpy(sub["lens"]).cuda(), None,
                           sub["bmm1_scale"], sub["bmm2_scale"], sub["k_scale"])
        outs.append(o)
        lses.append(l)
    out, lse = smla.merge(torch.stack(outs), torch.stack(lses))
    torch.cuda.synchronize()
    assert smla.smla_device_error() == 0
    T, H = w["q"].shape[:2]
    ref, ref_lse = oracle.fp64(oracle.Problem.from_workload(w))
    g = out.float().cpu().numpy().reshape(T * H, 512)
    live = ~np.isneginf(ref_lse)
    rowmax = np.abs(ref[live]).max(axis=1, keepdims=True)
    pairs = [(t, h) for t in range(T) for h in range(H)]
    e4m3 = e4m3_p_bound(w, [p for p, keep in zip(pairs, live) if keep])
    bound = np.maximum(TOL_FP64 * rowmax, e4m3) + 3 * bf16_ulp(ref[live])
    worst = float((np.abs(g[live] - ref[live]) / bound).max())
    print(f"decode shards + merge vs fp64 whole: worst {worst:.3f} of the bound")
    assert worst <= 1.0
    assert np.abs(lse.cpu().numpy().reshape(-1)[live] - ref_lse[live]).max() < 2e-3


def test_merge_full_size_sampled():
    """8 partial sets of the 64 x 128 batch shape; every 61st row checked."""
    S, T, H = 8, 64, 128
    parts, lses, lens = random_sets(2024, S, T, H, invalid=0.05, lens_zero=(5, 40))
    out, lse = smla.merge(parts.cuda(), torch.from_numpy(lses).cuda(), torch.from_numpy(lens).cuda())
    torch.cuda.synchronize()
    rows = np.arange(0, T * H, 61)
    t, h = rows // H, rows % H
    bits = parts.view(torch.int16).numpy().view(np.uint16)
    value, _, ref_lse = oracle.merge(oracle.MergeProblem(bits, lses, lens), pairs=np.stack([t, h], 1))
    g = out.float().cpu().numpy()[t, h]
    live = ~np.isneginf(ref_lse)
    assert np.all(out.view(torch.int16).cpu().numpy()[t[~live], h[~live]] == 0)
    scale = np.abs(parts.float().numpy()[:, t, h]).max(axis=(0, 2))
    bound = bf16_ulp(value) + 1e-6 * scale[:, None]
    assert (np.abs(g - value)[live] / bound[live]).max() <= 1.0
    assert np.abs(lse.cpu().numpy()[t, h][live] - ref_lse[live]).max() <= 1e-4
