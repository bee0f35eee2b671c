"""GPU parity of the decode over fp8_ds_mla rows (656 bytes: E4M3 latent codes,
four FP32 block scales, BF16 rope) against the FP64 definition of
``oracle/ds_mla.py``, through the C ABI.

Tolerance, from the kernel's arithmetic: every term is exact or FP32 except
one rounding to E4M3 of P * s_b / sigma_b per key and latent block (sigma_b
the running maximum of |s_b|), relative 2^-4 or absolute 2^-10 at most. In the
final frame (whose total is at least 448) that moves output element j of block
b by at most
    E_j = bmm2 * (sum_k w_k |V_kj| / 16 + 2^-10 / 448 * sigma_b * sum_k |code_kj|)
over the active keys k (w_k the definition's softmax weights, V the
dequantised latents, sigma_b the largest |s_b| of the token's keys). The test
takes max(0.02 * row max, E_j) plus one BF16 step of the output, and 1e-3 on
the base-2 LSE."""


import numpy as np
import pytest
import torch

from oracle import ds_mla
from sparse_mla_decode_gb300 import smla, workloads

pytestmark = pytest.mark.gpu


def q_values(w):
    """The query as float64 [T, H, 576] values (torch's E4M3 and BF16 decoders)."""
    lat = torch.from_numpy(w["q_latent"]).view(torch.float8_e4m3fn).to(torch.float64)
    rope = torch.from_numpy(w["q_rope"].view(np.int16)).view(torch.bfloat16).to(torch.float64)
    return torch.cat([lat, rope], dim=-1).numpy()


def one_pool(w):
    """The workload over the concatenation of its pools (the definition does
    not depend on how rows are split between pools)."""
    if len(w["pools"]) == 1:
        return w["pools"][0], w["indices"]
    rows0 = w["pools"][0].shape[0]
    idx = w["indices"].astype(np.int64).copy()
    second = np.arange(idx.shape[1]) >= w["pool_split"]
    idx[:, second] = np.where(idx[:, second] >= 0, idx[:, second] + rows0, -1)
    return np.concatenate(w["pools"]), idx.astype(np.int32)


def run_gpu(w, head_tile=0):
    dev = "cuda"
    ql = torch.from_numpy(w["q_latent"]).to(dev)
    qr = torch.from_numpy(w["q_rope"].view(np.int16)).view(torch.bfloat16).to(dev)
    pools = [torch.from_numpy(p).to(dev) for p in w["pools"]]
    idx = torch.from_numpy(w["indices"]).to(dev)
    lens = torch.from_numpy(w["lens"]).to(dev)
    sinks = None if w["sinks"] is None else torch.from_numpy(w["sinks"]).to(dev)
    out, lse = smla.decode_ds_mla(ql, qr, pools, idx, lens, sinks, w["bmm1_scale"], w["bmm2_scale"],
                                  pool_split=w["pool_split"], head_tile=head_tile)
    torch.cuda.synchronize()
    bits = smla.smla_device_error()
    assert bits & smla.DEV_TIMEOUT == 0
    return out.float().cpu().numpy(), out.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy(), bits


def bf16_ulp(x):
    a = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def compare(w, got, got_bits, got_lse):
    q = q_values(w)
    pool, indices = one_pool(w)
    ref, ref_lse = ds_mla.fp64(q, pool, indices, w["lens"], w["sinks"], w["bmm1_scale"], w["bmm2_scale"])
    T, H = q.shape[:2]
    W = indices.shape[1]
    worst = 0.0
    for t in range(T):
        n = min(max(int(w["lens"][t]), 0), W)
        cols = indices[t, :n]
        act = cols[(cols >= 0) & (cols < pool.shape[0])]
        if act.size == 0:
            assert np.all(got_bits[t] == 0), "an empty token's rows are +0.0"
            assert np.all(np.isneginf(got_lse[t])), "an empty token's LSE is -inf"
            continue
        kv = ds_mla.dequant_rows(pool[act])                                 # [A, 576]
        codes = torch.from_numpy(pool[act][:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        scales = pool[act][:, 512:528].copy().view("<f4").astype(np.float64)  # [A, 4]
        sigma = np.repeat(np.abs(scales).max(axis=0), 128)                   # [512]
        s = w["bmm1_scale"] * (q[t] @ kv.T)                                  # [H, A]
        top = s.max(axis=1)
        if w["sinks"] is not None:
            top = np.maximum(top, w["sinks"].astype(np.float64))
        e = np.exp(s - top[:, None])
        den = e.sum(axis=1) + (0.0 if w["sinks"] is None else np.exp(w["sinks"].astype(np.float64) - top))
        wk = e / den[:, None]                                                # [H, A]
        e_j = w["bmm2_scale"] * (wk @ np.abs(kv[:, :512]) / 16.0 +
                                 (2.0 ** -10 / 448.0) * sigma * np.abs(codes).sum(axis=0)[None, :])
        rowmax = np.abs(ref[t]).max(axis=1, keepdims=True)
        bound = np.maximum(0.02 * rowmax, e_j) + bf16_ulp(ref[t])
        err = np.abs(got[t] - ref[t])
        worst = max(worst, float((err / bound).max()))
        assert np.abs(got_lse[t] - ref_lse[t]).max() <= 1e-3, f"token {t}: lse"
    assert worst <= 1.0, f"worst error at {worst:.3f} of the bound"
    return worst


CASES = [
    # tokens, heads, width, pool rows, holes, sinks, lens, two pools (split)
    (2, 32, 300, 600, 0.1, True, [300, 77], None),        # ragged: 128 + 128 + 44
    (3, 64, 1000, 4000, 0.05, False, [1000, 129, 0], None),  # an empty token
    (1, 32, 128, 500, 0.0, True, None, None),              # one full chunk
    (2, 128, 2048, 10000, 0.05, True, [2048, 1500], None),
    (2, 32, 384, 400, 0.05, True, [384, 200], 128),        # two pools: 128 window + top-k
    (2, 64, 700, 900, 0.1, True, [700, 5], 256),           # two pools, 64 heads, a token inside chunk 0
    (1, 64, 1, 10, 0.0, True, None, None),                 # one key
]


@pytest.mark.parametrize("case", CASES, ids=[f"t{c[0]}_h{c[1]}_w{c[2]}" + ("_2p" if c[7] else "") for c in CASES])
def test_ds_mla_rows_match_the_definition(case):
    """Each head tile the shape allows (32, and 64 where H is a multiple of
    64) against the definition; the two tiles compute the same arithmetic in
    the same order, so their outputs agree bit for bit."""
    T, H, W, rows, holes, sinks, lens, split = case
    w = workloads.ds_mla_small("ds", seed=T * 1000 + W, tokens=T, heads=H, width=W, pool_rows=rows, holes=holes,
                               lens=lens, sinks=sinks, two_pools=split is not None, pool_split=split or 0)
    results = {}
    for tile in (32, 64) if H % 64 == 0 else (32,):
        got, bits, lse, dev_bits = run_gpu(w, head_tile=tile)
        assert dev_bits == 0
        print(case, "tile", tile, "worst", compare(w, got, bits, lse))
        results[tile] = (bits, lse)
    if 64 in results:
        assert np.array_equal(results[32][0], results[64][0]), "64-head tiles: the same bits as 32-head tiles"
        assert np.array_equal(results[32][1], results[64][1])


@pytest.mark.parametrize("heads,tile", [(32, 32), (64, 64)])
def test_rising_block_scales_rescale_the_accumulated_blocks(heads, tile):
    """Rows whose scales grow with the row number, gathered in increasing
    order: every chunk raises each block's largest scale, so the accumulated
    output blocks are rescaled chunk after chunk (and each block differently)."""
    w = workloads.ds_mla_small("rising", seed=5, tokens=2, heads=heads, width=1024, pool_rows=1024, sinks=True)
    pool = w["pools"][0]
    r = np.arange(pool.shape[0], dtype=np.float64)
    scales = np.stack([2.0 ** (r / 64.0 - 12 + b) for b in range(4)], axis=1).astype("<f4")
    pool[:, 512:528] = scales.view(np.uint8).reshape(-1, 16)
    w["indices"] = np.tile(np.arange(1024, dtype=np.int32), (2, 1))
    w["lens"] = np.array([1024, 700], np.int32)
    got, bits, lse, _ = run_gpu(w, head_tile=tile)
    print("worst", compare(w, got, bits, lse))


@pytest.mark.parametrize("heads,tile", [(32, 32), (64, 64)])
def test_index_beyond_the_pool_is_masked_and_flagged(heads, tile):
    w = workloads.ds_mla_small("oob", seed=9, tokens=1, heads=heads, width=64, pool_rows=100)
    w["indices"][0, 10] = 100
    w["indices"][0, 11] = 1 << 30
    got, bits, lse, dev_bits = run_gpu(w, head_tile=tile)
    assert dev_bits == smla.DEV_INDEX_RANGE
    compare(w, got, bits, lse)  # the definition treats them as holes


def test_output_scale_and_repeated_calls():
    w = workloads.ds_mla_small("scale", seed=3, tokens=2, heads=32, width=500, pool_rows=800, bmm2_scale=0.375)
    a = run_gpu(w)
    b = run_gpu(w)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    compare(w, *a[:3])


def test_zero_tokens_and_zero_width():
    w = workloads.ds_mla_small("empty", seed=4, tokens=2, heads=32, width=0, pool_rows=10)
    got, bits, lse, _ = run_gpu(w)
    assert np.all(bits == 0) and np.all(np.isneginf(lse))
    ql = torch.zeros((0, 32, 512), dtype=torch.uint8, device="cuda")
    qr = torch.zeros((0, 32, 64), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((4, 656), dtype=torch.uint8, device="cuda")
    idx = torch.zeros((0, 8), dtype=torch.int32, device="cuda")
    lens = torch.zeros((0,), dtype=torch.int32, device="cuda")
    smla.decode_ds_mla(ql, qr, [pool], idx, lens)
    torch.cuda.synchronize()
    assert smla.smla_device_error() == 0


def test_batch_shape_in_both_head_tiles():
    """The 64 x 128 x 2048 batch shape, half of each token's rows from a
    shared hot set, against the definition: 64-head tiles (the library's
    choice here: 128 CTAs, one wave) and 32-head tiles (256 CTAs, more than
    one wave), bit for bit the same."""
    w = workloads.ds_mla_batch(seed=21, pool_rows=100_000, hot_rows=5000)
    assert smla.smla_ds_mla_head_tile(64, 128) == 64
    got, bits, lse, dev_bits = run_gpu(w)
    assert dev_bits == 0
    print("worst", compare(w, got, bits, lse))
    _, bits32, lse32, dev_bits = run_gpu(w, head_tile=32)
    assert dev_bits == 0
    assert np.array_equal(bits, bits32) and np.array_equal(lse, lse32)
