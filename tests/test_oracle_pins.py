"""Pins of the CPU oracle to facts outside itself.

Each test checks one part of ``oracle/`` against something it does not share
code with: torch's E4M3 / BF16 codecs (library routines), torch's
scaled-dot-product attention in float64 (the special case of the decode with
every gathered row active), closed forms, and invariants of the definition
(DeepSeek-V4.1 ``sparse_mla_cute`` page, "What this module computes"; Kimi K3.1
``attn_sparse`` page, module docstring and ``SparseDcpDecode.merge``).  A
plausible slip in the oracle -- a dropped term, a wrong sign or index, a
transposed operand, the P anchor at the wrong maximum -- fails one of them.
"""

import math

import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_mla_decode_gb300 import workloads

LOG2E = 1.0 / math.log(2.0)


def dec(b):
    """E4M3 bytes -> float64 through torch (the library decoder)."""
    t = torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


# ----------------------------------------------------------------- codecs


def test_e4m3_decode_every_byte_matches_torch():
    ref = dec(np.arange(256, dtype=np.uint8))
    got = np.array([oracle.e4m3_to_double(b) for b in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def _e4m3_grid():
    finite = dec(np.arange(0, 0x7F, dtype=np.uint8))  # 0 .. 448
    mids = (finite[1:] + finite[:-1]) / 2
    pts = np.concatenate([finite, mids])
    f32 = pts.astype(np.float32)
    up = np.nextafter(f32, np.float32(np.inf))
    dn = np.nextafter(f32, np.float32(-np.inf))
    rng = np.random.default_rng(7)
    rand = rng.uniform(0, 470, 20000).astype(np.float32)
    tiny = rng.uniform(0, 2 ** -5, 5000).astype(np.float32)
    g = np.concatenate([f32, up, dn, rand, tiny])
    return np.concatenate([g, -g])


def test_e4m3_encode_rn_matches_torch_in_range():
    g = _e4m3_grid()
    g = g[np.abs(g) < 464.0]  # torch's cast is RN without saturation; equal below 464
    ref = torch.from_numpy(g).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(x) for x in g], np.uint8)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(g[i]), int(ref[i]), int(got[i])) for i in bad[:5]]


def test_e4m3_encode_saturates_and_nan():
    # satfinite: anything at or beyond the largest finite value maps to +-448
    for x in [448.0, 449.0, 464.0, 500.0, 1e30, float("inf")]:
        assert oracle.e4m3_from_float(x) == 0x7E
        assert oracle.e4m3_from_float(-x) == 0xFE
    assert oracle.e4m3_from_float(float("nan")) & 0x7F == 0x7F
    assert oracle.e4m3_from_float(2.0 ** -10) == 0x00  # tie to even (0)
    assert oracle.e4m3_from_float(3 * 2.0 ** -10) == 0x02  # tie to even (2)


def test_bf16_rn_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(50000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 50000),
        np.array([0.0, -0.0, 1.0, 3.4e38, -3.4e38, 1e-40], np.float32),
    ]).astype(np.float32)
    # exact ties: a BF16 value plus half an ULP
    base = (rng.integers(0, 1 << 16, 2000).astype(np.uint32) << 16) | 0x8000
    x = np.concatenate([x, base.view(np.float32)])
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_float(v) for v in x], np.uint16)
    assert np.array_equal(ref, got)


# ------------------------------------------------------- the definition


def _sdpa_reference(w, t, h):
    """Library evaluation of one (token, head): torch SDPA in float64 over the
    gathered active rows (numpy indexing), the sink as an extra key whose bias
    equals the sink and whose value row is zero."""
    D = w["q"].shape[2]
    W = w["indices"].shape[1]
    n = max(0, min(int(w["lens"][t]), W))
    rows = []
    for c in range(n):
        r = int(w["indices"][t, c])
        pool = 1 if (len(w["pools"]) == 2 and c >= w["pool_split"]) else 0
        if r < 0 or r >= w["pools"][pool].shape[0]:
            continue
        rows.append(w["pools"][pool][r])
    if not rows:
        return np.zeros(512), -np.inf
    kv = torch.from_numpy(dec(np.stack(rows)))  # [n, D]
    q = torch.from_numpy(dec(w["q"][t, h]))[None, None, None, :]  # [1,1,1,D]
    k = kv[None, None]  # [1,1,n,D]
    v = kv[None, None, :, :512]
    bias = torch.zeros(1, 1, 1, kv.shape[0], dtype=torch.float64)
    if w["sinks"] is not None:
        k = torch.cat([k, torch.zeros(1, 1, 1, D, dtype=torch.float64)], dim=2)
        v = torch.cat([v, torch.zeros(1, 1, 1, 512, dtype=torch.float64)], dim=2)
        bias = torch.cat([bias, torch.full((1, 1, 1, 1), float(w["sinks"][h]), dtype=torch.float64)], -1)
    out = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=bias, scale=float(w["bmm1_scale"]))
    logits = (q[0, 0] @ k[0, 0].T)[0] * w["bmm1_scale"] + bias[0, 0, 0]
    lse = torch.logsumexp(logits, dim=0).item()
    return out[0, 0, 0].numpy() * w["bmm2_scale"] * w["k_scale"], lse * LOG2E


CASES = [
    dict(name="dense", seed=11, tokens=2, heads=16, width=40, head_dim=576),
    dict(name="holes_lens", seed=12, tokens=3, heads=16, width=50, head_dim=576, holes=0.3,
         lens=[50, 17, 33]),
    dict(name="sinks_512", seed=13, tokens=2, heads=16, width=30, head_dim=512, sinks=True,
         k_scale=0.05, bmm2_scale=0.5),
    dict(name="two_pools", seed=14, tokens=2, heads=16, width=37, head_dim=512, two_pools=True,
         pool_split=13, holes=0.1, sinks=True),
    dict(name="duplicates", seed=15, tokens=1, heads=16, width=64, head_dim=576,
         pool_rows=20, duplicates=True),
]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_fp64_matches_library_attention(case):
    w = workloads.small(**case)
    prob = oracle.Problem.from_workload(w)
    out, lse = oracle.fp64(prob)
    T, H = w["q"].shape[:2]
    for t in range(T):
        for h in range(H):
            ref_out, ref_lse = _sdpa_reference(w, t, h)
            i = t * H + h
            scale = max(1e-300, np.abs(ref_out).max())
            assert np.abs(out[i] - ref_out).max() <= 1e-12 * scale
            assert abs(lse[i] - ref_lse) <= 1e-12 * max(1.0, abs(ref_lse))


def test_single_active_key_returns_the_row():
    w = workloads.small("one", seed=21, tokens=1, heads=16, width=8, head_dim=576, lens=[8])
    w["indices"][0, :] = -1
    w["indices"][0, 5] = 77
    w["k_scale"], w["bmm2_scale"] = 0.25, 0.5
    prob = oracle.Problem.from_workload(w)
    out, lse = oracle.fp64(prob)
    v = dec(w["pools"][0][77, :512]) * 0.125
    s = dec(w["q"][0]) @ dec(w["pools"][0][77]) * w["bmm1_scale"]
    assert np.array_equal(out, np.broadcast_to(v, out.shape))
    assert np.allclose(lse, s * LOG2E, rtol=0, atol=1e-12)
    # emulating mode: P = 448 exactly, l = 448, so out = BF16(V * scale)
    val, bits, lse_e = oracle.emulate(prob, splits=3, chunk=2)
    ref_bits = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(bits.view(np.int16), np.broadcast_to(ref_bits, bits.shape))
    assert np.allclose(lse_e, s * LOG2E, atol=1e-5)


def test_equal_scores_give_the_mean_row():
    w = workloads.small("eq", seed=22, tokens=1, heads=16, width=100, head_dim=576, holes=0.2)
    w["q"][:] = 0  # every score 0
    prob = oracle.Problem.from_workload(w)
    out, lse = oracle.fp64(prob)
    act = w["indices"][0][w["indices"][0] >= 0]
    mean = dec(w["pools"][0][act, :512]).mean(axis=0)
    assert np.allclose(out, mean[None], rtol=0, atol=1e-14)
    assert np.allclose(lse, math.log2(act.size), atol=1e-13)
    val, bits, lse_e = oracle.emulate(prob, splits=2, chunk=32)
    assert np.allclose(val, mean[None], rtol=0, atol=2e-6 * np.abs(mean).max())
    assert np.allclose(lse_e, math.log2(act.size), atol=1e-6)


def test_permuting_columns_changes_nothing():
    w = workloads.small("perm", seed=23, tokens=2, heads=16, width=90, head_dim=576, holes=0.15,
                        sinks=True)
    prob = oracle.Problem.from_workload(w)
    out, lse = oracle.fp64(prob)
    rng = np.random.default_rng(5)
    for t in range(2):
        w["indices"][t] = w["indices"][t][rng.permutation(90)]
    out2, lse2 = oracle.fp64(oracle.Problem.from_workload(w))
    assert np.allclose(out, out2, rtol=0, atol=1e-12 * np.abs(out).max())
    assert np.allclose(lse, lse2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("sinks", [False, True])
def test_empty_tokens_give_zeros_and_minus_inf(sinks):
    w = workloads.small("empty", seed=24, tokens=4, heads=16, width=20, head_dim=576,
                        lens=[0, 20, -5, 7], sinks=sinks)
    w["indices"][1, :] = -1  # all holes
    w["indices"][3, :7] = -1  # holes inside the count, active ones past it
    prob = oracle.Problem.from_workload(w)
    out, lse = oracle.fp64(prob)
    val, bits, lse_e = oracle.emulate(prob, splits=2, chunk=8)
    assert np.all(out == 0) and not np.any(np.signbit(out))
    assert np.all(np.isneginf(lse))
    assert np.all(bits == 0)
    assert np.all(np.isneginf(lse_e))


def test_sink_removes_weight_in_closed_form():
    base = workloads.small("sink", seed=25, tokens=2, heads=16, width=60, head_dim=576,
                           holes=0.1, sinks=True)
    with_sink = oracle.fp64(oracle.Problem.from_workload(base))
    no = dict(base)
    no["sinks"] = None
    out0, lse0 = oracle.fp64(oracle.Problem.from_workload(no))
    sinks = np.tile(base["sinks"].astype(np.float64), 2)
    # exp(lse) is the denominator; a sink adds exp(sink) to it and nothing to the sum
    den0 = lse0 / LOG2E
    frac = 1.0 / (1.0 + np.exp(sinks - den0))
    assert np.allclose(with_sink[0], out0 * frac[:, None], rtol=1e-12, atol=1e-15)
    assert np.allclose(with_sink[1], np.logaddexp(den0, sinks) * LOG2E, atol=1e-12)


# ---------------------------------------------------- the emulated datapath


@pytest.mark.parametrize("splits,chunk", [(1, 128), (2, 16), (3, 7), (4, 1), (7, 5)])
def test_online_softmax_and_merge_equal_the_definition(splits, chunk):
    """With P unrounded and no FP32 steps, any partition into chunks and splits
    must reproduce the plain definition (the running-max rescale and the merge
    weights cancel exactly)."""
    w = workloads.small("merge", seed=31, tokens=3, heads=16, width=70, head_dim=576, holes=0.2,
                        lens=[70, 3, 41], sinks=True)
    prob = oracle.Problem.from_workload(w)
    out, lse = oracle.fp64(prob)
    val, _, lse_e = oracle.emulate(prob, splits, chunk, flags=oracle.EXACT | oracle.NO_P_ROUNDING)
    assert np.abs(val - out).max() <= 1e-12 * np.abs(out).max()
    assert np.abs(lse_e - lse).max() <= 1e-12 * np.abs(lse).max()


def test_p_anchors_at_the_running_max():
    """Two active keys in two one-key chunks, the second scoring far higher.
    Against the running max both P are exactly 448, so the result is the exact
    softmax; anchored at the final maximum, the first P would be rounded."""
    w = workloads.small("anchor", seed=32, tokens=1, heads=16, width=2, head_dim=576)
    w["q"][:] = 0
    q = np.zeros(576, np.float32)
    q[0] = 1.0
    w["q"][0, :] = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    pool = w["pools"][0]
    pool[:2, 0] = torch.tensor([1.0, 1.5]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    w["indices"][0] = [0, 1]
    w["bmm1_scale"] = 1.0
    prob = oracle.Problem.from_workload(w)
    v0, v1 = dec(pool[0, :512]), dec(pool[1, :512])
    s0, s1 = 1.0 * LOG2E, 1.5 * LOG2E
    alpha = 2.0 ** (np.float32(s0) - np.float32(s1))
    exact = (alpha * v0 + v1) / (alpha + 1)
    val, _, _ = oracle.emulate(prob, splits=1, chunk=1)
    assert np.allclose(val[0], exact, rtol=0, atol=1e-5 * np.abs(exact).max())
    # one chunk: the first P is rounded to E4M3 (torch's codec) before PV
    p0 = float(torch.tensor([448.0 * alpha], dtype=torch.float32).to(torch.float8_e4m3fn).float())
    assert p0 != np.float32(448.0 * alpha)  # the test is only meaningful if rounding bites
    quantised = (p0 * v0 + 448.0 * v1) / (448.0 * alpha + 448.0)
    val1, _, _ = oracle.emulate(prob, splits=1, chunk=2)
    assert np.allclose(val1[0], quantised, rtol=0, atol=1e-5 * np.abs(quantised).max())
    assert np.abs(val1[0] - exact).max() > 1e-3 * np.abs(exact).max()


def test_tie_window_bound_covers_both_codes_of_a_midpoint_p():
    """A P that lands on a rounding midpoint of E4M3 (46, between the codes 44
    and 48) may take either code under the datapath's FP32 arithmetic (Kimi
    K3.1 attn_sparse page, "Precision": FP32 logits of FP8 products in an
    unspecified order, a fast exp2). Two keys: the first scores the maximum (P
    = 448), the second is placed by bmm1_scale at P = 448 * 2^log2(46/448). The
    two codes move the output by 4 * V_2 * out_scale / l in closed form, and
    the emulation's tie bound is exactly that spread."""
    w = workloads.small("tie", seed=31, tokens=1, heads=16, width=2, head_dim=576, pool_rows=64, lens=[2])
    w["indices"][0] = [3, 9]
    q, k1, k2 = dec(w["q"][0, 0]), dec(w["pools"][0][3]), dec(w["pools"][0][9])
    s1, s2 = q @ k1, q @ k2
    if s1 < s2:
        w["indices"][0] = [9, 3]
        s1, s2, k1, k2 = s2, s1, k2, k1
    w["bmm1_scale"] = math.log2(46.0 / 448.0) / ((s2 - s1) * LOG2E)
    w["bmm2_scale"], w["k_scale"] = 0.5, 1.0
    prob = oracle.Problem.from_workload(w)
    val, _, _, tie = oracle.emulate(prob, 1, 128, pairs=[(0, 0)], ties=True)
    up, _, _ = oracle.emulate(prob, 1, 128, pairs=[(0, 0)], flags=oracle.P_UP)
    down, _, _ = oracle.emulate(prob, 1, 128, pairs=[(0, 0)], flags=oracle.P_DOWN)
    l = 448.0 + 46.0
    spread = 4.0 * k2[:512] * 0.5 / l
    # the outputs carry FP32 roundings of values up to ~0.5 (2^-24 each)
    assert np.allclose(up[0] - down[0], spread, rtol=0, atol=2e-7)
    assert np.allclose(tie[0], np.abs(spread), rtol=1e-6, atol=0)
    assert np.all((val[0] == up[0]) | (val[0] == down[0]))


@pytest.mark.parametrize("splits,chunk", [(1, 256), (3, 128), (2, 64)])
def test_tie_bound_is_zero_without_midpoints_and_covers_the_other_codes(splits, chunk):
    """On random workloads the codes of the window's two edges differ only
    where the tie bound is positive, and never by more than it."""
    w = workloads.small("ties", seed=32 + splits, tokens=3, heads=32, width=700, head_dim=576, pool_rows=4096,
                        holes=0.05, sinks=True, lens=[700, 333, 9])
    prob = oracle.Problem.from_workload(w)
    val, _, _, tie = oracle.emulate(prob, splits, chunk, ties=True)
    up, _, _ = oracle.emulate(prob, splits, chunk, flags=oracle.P_UP)
    down, _, _ = oracle.emulate(prob, splits, chunk, flags=oracle.P_DOWN)
    gap = np.maximum(np.abs(up - val), np.abs(down - val))
    assert np.all(gap <= tie * (1 + 1e-6) + 1e-7 * np.abs(val).max())
    quiet = tie.max(axis=1) == 0
    assert quiet.mean() > 0.5  # most rows have no P near a midpoint
    assert np.array_equal(up[quiet], val[quiet]) and np.array_equal(down[quiet], val[quiet])


def test_one_chunk_matches_a_float32_library_evaluation():
    """One split, one chunk: the datapath is P = E4M3(2^(s2 - m + log2 448))
    with FP32 logits, sums of the unrounded P, FP32 PV, one BF16 rounding --
    evaluated here with torch float32 ops and torch's E4M3 cast."""
    w = workloads.small("chunk", seed=33, tokens=2, heads=16, width=100, head_dim=576, holes=0.1)
    prob = oracle.Problem.from_workload(w)
    val, bits, lse = oracle.emulate(prob, splits=1, chunk=128)
    for t in range(2):
        act = w["indices"][t][w["indices"][t] >= 0]
        kv = torch.from_numpy(dec(w["pools"][0][act]))
        q = torch.from_numpy(dec(w["q"][t]))
        logits = (q @ kv.T).to(torch.float32)  # exact sums rounded once
        s2 = logits * torch.tensor(w["bmm1_scale"] * LOG2E, dtype=torch.float32)
        m = s2.max(dim=1, keepdim=True).values
        p = torch.exp2(s2 - (m - torch.tensor(math.log2(448.0), dtype=torch.float32)))
        l = p.sum(dim=1, keepdim=True)
        p8 = p.to(torch.float8_e4m3fn).to(torch.float64)
        acc = (p8 @ kv[:, :512]).to(torch.float32)
        ref = (acc * (1.0 / l)).to(torch.float64).numpy()
        got = val[t * 16:(t + 1) * 16]
        assert np.abs(got - ref).max() <= 2e-6 * np.abs(ref).max()
        ref_lse = (m[:, 0] - math.log2(448.0) + torch.log2(l[:, 0])).numpy()
        assert np.abs(lse[t * 16:(t + 1) * 16] - ref_lse).max() <= 1e-5


# ------------------------------------------------ LSE merge of partial sets
# (Kimi K3.1 mla/dcp page, DcpValue: weights exp2(lse - max) / sum, FP32 merge
# of the BF16 rows, one BF16 rounding; empty sources weigh nothing.)


def _column_subset(w, t_cols):
    """The workload with only the columns in ``t_cols[t]`` kept (others -1)."""
    sub = dict(w)
    sub["indices"] = np.full_like(w["indices"], -1)
    for t, cols in enumerate(t_cols):
        cols = np.asarray(cols, dtype=np.int64)
        sub["indices"][t, cols] = w["indices"][t, cols]
    return sub


@pytest.mark.parametrize("layout", ["blocks", "interleaved", "with_empty_part"])
def test_merge_of_key_disjoint_parts_equals_the_definition(layout):
    """Decoding disjoint column subsets separately and merging the parts by
    their LSEs reassembles the decode of all columns (the softmax over a union
    of keys): pins the weights' base, sign and normalisation to the decode
    definition."""
    w = workloads.small("merge_pin", seed=404, tokens=2, heads=16, width=60, head_dim=576,
                        pool_rows=300, holes=0.1, lens=[60, 45])
    W = w["indices"].shape[1]
    if layout == "blocks":
        parts = [list(range(0, 20)), list(range(20, 41)), list(range(41, W))]
    elif layout == "interleaved":
        parts = [list(range(s, W, 3)) for s in range(3)]
    else:
        parts = [list(range(0, 30)), [], list(range(30, W))]
    whole = oracle.Problem.from_workload(w)
    ref, ref_lse = oracle.fp64(whole)
    outs, lses = [], []
    for cols in parts:
        sub = oracle.Problem.from_workload(_column_subset(w, [cols, cols]))
        o, l = oracle.fp64(sub)
        outs.append(o)
        lses.append(l)
    outs = np.stack(outs)  # [S, T*H, 512]
    lses = np.stack(lses)  # [S, T*H]
    for i in range(ref.shape[0]):
        got, got_lse = oracle.merge_f64(outs[:, i], lses[:, i])
        np.testing.assert_allclose(got, ref[i], rtol=1e-12, atol=1e-14)
        assert abs(got_lse - ref_lse[i]) < 1e-12


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_value(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


def test_merge_with_one_valid_source_passes_it_through():
    rng = np.random.default_rng(1)
    parts = _bf16_bits(rng.standard_normal((4, 1, 2, 512)))
    lses = np.array([[[-np.inf, 3.0]], [[2.5, np.nan]], [[np.nan, -np.inf]], [[np.inf, np.inf]]], np.float32)
    _, bits, lse = oracle.merge(oracle.MergeProblem(parts, lses))
    assert np.array_equal(bits[0], parts[1, 0, 0]) and lse[0] == 2.5
    assert np.array_equal(bits[1], parts[0, 0, 1]) and lse[1] == 3.0


def test_merge_of_equal_lses_is_the_mean_row():
    rng = np.random.default_rng(2)
    parts = _bf16_bits(rng.standard_normal((5, 2, 3, 512)))
    lses = np.full((5, 2, 3), 7.25, np.float32)
    value, _, lse = oracle.merge(oracle.MergeProblem(parts, lses))
    mean = _bf16_value(parts).astype(np.float64).mean(axis=0).reshape(-1, 512)
    np.testing.assert_allclose(value, mean, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse, 7.25 + math.log2(5.0), rtol=0, atol=1e-12)


def test_merge_weights_in_closed_form():
    """Two sources: out = (a * 2^la + b * 2^lb) / (2^la + 2^lb)."""
    rng = np.random.default_rng(3)
    parts = _bf16_bits(rng.standard_normal((2, 1, 1, 512)))
    la, lb = 1.0, -2.5
    lses = np.array([[[la]], [[lb]]], np.float32)
    value, _, lse = oracle.merge(oracle.MergeProblem(parts, lses))
    a, b = _bf16_value(parts[0, 0, 0]).astype(np.float64), _bf16_value(parts[1, 0, 0]).astype(np.float64)
    expect = (a * 2.0 ** la + b * 2.0 ** lb) / (2.0 ** la + 2.0 ** lb)
    np.testing.assert_allclose(value[0], expect, rtol=1e-14, atol=1e-16)
    assert abs(lse[0] - math.log2(2.0 ** la + 2.0 ** lb)) < 1e-12


def test_merge_is_shift_and_permutation_invariant():
    rng = np.random.default_rng(4)
    parts = _bf16_bits(rng.standard_normal((6, 2, 2, 512)))
    lses = (np.round(rng.uniform(-5, 5, (6, 2, 2)) * 1024) / 1024).astype(np.float32)  # + 16 is exact
    v0, b0, l0 = oracle.merge(oracle.MergeProblem(parts, lses))
    v1, b1, l1 = oracle.merge(oracle.MergeProblem(parts, lses + np.float32(16.0)))
    np.testing.assert_allclose(v1, v0, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(l1, l0 + 16.0, rtol=0, atol=1e-9)
    perm = rng.permutation(6)
    v2, _, l2 = oracle.merge(oracle.MergeProblem(parts[perm], lses[perm]))
    np.testing.assert_allclose(v2, v0, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(l2, l0, rtol=0, atol=1e-12)


def test_merge_empty_rows_are_zero_and_minus_inf():
    rng = np.random.default_rng(5)
    parts = _bf16_bits(rng.standard_normal((3, 3, 1, 512)))
    lses = rng.uniform(-2, 2, (3, 3, 1)).astype(np.float32)
    lses[:, 1, 0] = -np.inf  # every source empty
    value, bits, lse = oracle.merge(oracle.MergeProblem(parts, lses, lens=np.array([5, 5, 0], np.int32)))
    for i in (1, 2):  # all sources empty; token count 0
        assert np.all(bits[i] == 0) and np.all(value[i] == 0.0) and lse[i] == -np.inf
    assert np.isfinite(lse[0])


# -------------------------------- MXFP4 quantisation of the indexer query
# (Kimi K3.1 dsa_indexer_mxfp4 page: UE8M0 scale 2^ceil(log2(amax / 6)) per 32
# values, E2M1 codes with the even element in the low nibble.)

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_grid_round_trips_and_ties_go_to_even_codes():
    for code in range(16):
        v = oracle.e2m1_to_double(code)
        assert abs(v) == E2M1_GRID[code & 7] and (v < 0) == (code >= 8 and code != 8)
        if code != 8:  # -0 decodes to 0 and re-encodes to +0 (0.0 has no sign)
            assert oracle.e2m1_from_float(v) == code
    # midpoints between neighbours: the code with mantissa bit 0 wins
    for lo in range(7):
        mid = (E2M1_GRID[lo] + E2M1_GRID[lo + 1]) / 2
        even = lo if lo % 2 == 0 else lo + 1
        assert oracle.e2m1_from_float(mid) == even
        assert oracle.e2m1_from_float(-mid) == 8 | even
    assert oracle.e2m1_from_float(6.5) == 7 and oracle.e2m1_from_float(1e30) == 7  # saturating
    assert oracle.e2m1_from_float(-1e-6) == 8  # the sign of a zero result is kept


def test_e2m1_rounds_to_the_nearest_grid_value():
    rng = np.random.default_rng(6)
    grid = np.array(E2M1_GRID)
    for x in rng.uniform(-7, 7, 3000).astype(np.float32):
        v = oracle.e2m1_to_double(oracle.e2m1_from_float(float(x)))
        a = min(abs(float(x)), 6.0)
        assert abs(abs(v) - a) <= np.min(np.abs(grid - a)) + 1e-12


def _mxfp4_inputs(seed, T=3, H=5):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((T, H, 128)) * rng.uniform(1e-3, 1e3, (T, H, 1))).astype(np.float32)
    q[0, 0, 32:64] = 0.0  # an all-zero block
    q[0, 1, 0:32] = 6.0 * 2.0 ** -3  # amax exactly 6 * 2^-3
    q[0, 1, 32:64] = np.float32(6.0 * 2.0 ** -3) * np.float32(1 + 2 ** -20)  # just above
    w = rng.standard_normal((T, H)).astype(np.float32)
    return q, w


def test_mxfp4_scale_is_the_smallest_power_of_two_covering_the_block():
    q, w = _mxfp4_inputs(7)
    packed, scale, _ = oracle.mxfp4_q_quant(q, w, 0.5, 8)
    T, H, _ = q.shape
    for t in range(T):
        for h in range(H):
            for b in range(4):
                e = int((int(scale[t, h]) >> (8 * b)) & 0xFF) - 127
                amax = float(np.abs(q[t, h, 32 * b:32 * b + 32]).max())
                if amax <= 6.0 * 2.0 ** -126:
                    assert e == -126
                else:
                    assert amax <= 6.0 * 2.0 ** e and amax > 6.0 * 2.0 ** (e - 1)
    assert (int(scale[0, 1]) & 0xFF) - 127 == -3 and ((int(scale[0, 1]) >> 8) & 0xFF) - 127 == -2


def test_mxfp4_dequantised_values_are_within_half_a_grid_step():
    q, w = _mxfp4_inputs(8)
    packed, scale, _ = oracle.mxfp4_q_quant(q, w, 1.0, 5)
    grid = np.array(E2M1_GRID)
    T, H, _ = q.shape
    for t in range(T):
        for h in range(H):
            for i in range(128):
                byte = int(packed[t, h, i // 2])
                code = byte & 0xF if i % 2 == 0 else byte >> 4  # even element in the low nibble
                e = int((int(scale[t, h]) >> (8 * (i // 32))) & 0xFF) - 127
                y = float(q[t, h, i]) / 2.0 ** e
                back = oracle.e2m1_to_double(code)
                gap = np.min(np.abs(grid - min(abs(y), 6.0)))
                assert abs(abs(back) - min(abs(y), 6.0)) <= gap + 1e-12
                assert back == 0.0 or np.sign(back) == np.sign(y)


def test_mxfp4_zero_blocks_weights_and_padding():
    q, w = _mxfp4_inputs(9, T=2, H=3)
    packed, scale, w_out = oracle.mxfp4_q_quant(q, w, 0.125, 8)
    assert ((int(scale[0, 0]) >> 8) & 0xFF) == 1 and np.all(packed[0, 0, 16:32] == 0)  # zero block: 2^-126
    np.testing.assert_array_equal(w_out[:, :3], w * np.float32(0.125))
    assert np.all(packed[:, 3:] == 0) and np.all(scale[:, 3:] == 0) and np.all(w_out[:, 3:] == 0)


# ------------------- value projection and sigmoid gate (mla/dcp, DcpValue)


def _bf(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def _value_gate_inputs(seed, T=3, H=2):
    rng = np.random.default_rng(seed)
    latent = _bf(rng.standard_normal((T, H, 512)) * 0.5)
    w = _bf(rng.standard_normal((H, 512, 128)) * 0.05)
    gate = _bf(rng.standard_normal((T, H * 128)) * 2.0)
    return latent, w, gate


def test_value_gate_matches_a_library_matmul():
    """The oracle's loops against numpy's float64 matmul of the same BF16
    values, with the roundings and the sigmoid applied on top."""
    latent, w, gate = _value_gate_inputs(21)
    value, bits = oracle.value_gate(latent, w, gate)
    acc = np.einsum("thj,hjv->thv", _val(latent), _val(w))
    rounded = _val(_bf(acc.astype(np.float32)))
    expect = (rounded * (1.0 / (1.0 + np.exp(-_val(gate).reshape(rounded.shape))))).reshape(value.shape)
    np.testing.assert_allclose(value, expect, rtol=1e-12, atol=1e-14)
    assert np.array_equal(bits, _bf(expect.astype(np.float32)))


def test_value_gate_with_an_identity_projection_is_the_gated_latent():
    latent, _, gate = _value_gate_inputs(22, T=2, H=3)
    w = np.zeros((3, 512, 128), np.float32)
    for v in range(128):
        w[:, 2 * v, v] = 1.0  # v reads latent 2v
    value, _ = oracle.value_gate(latent, _bf(w), gate)
    lat = _val(latent)[:, :, 0:256:2].reshape(2, 3 * 128)
    np.testing.assert_allclose(value, lat / (1.0 + np.exp(-_val(gate))), rtol=1e-14)


def test_value_gate_saturated_gates_and_empty_tokens():
    latent, w, gate = _value_gate_inputs(23)
    gate = _bf(np.where(np.arange(3 * 0 + 2 * 128)[None, :] % 2 == 0, 40.0, -40.0) * np.ones((3, 1)))
    value, bits = oracle.value_gate(latent, w, gate, lens=np.array([5, 0, 1], np.int32))
    acc = np.einsum("thj,hjv->thv", _val(latent), _val(w)).reshape(3, 256)
    rounded = _val(_bf(acc.astype(np.float32)))
    np.testing.assert_allclose(value[[0, 2]][:, ::2], rounded[[0, 2]][:, ::2], rtol=1e-12)  # sigmoid(40) = 1 - 4e-18
    assert np.all(np.abs(value[[0, 2]][:, 1::2]) <= np.abs(rounded[[0, 2]][:, 1::2]) * 1e-17)  # sigmoid(-40)
    assert np.all(value[1] == 0.0) and np.all(bits[1] == 0)  # a token of count 0


@pytest.mark.parametrize("make,low", [(workloads.tiny, 0.022), (workloads.verify_rows, 0.022),
                                      (workloads.two_pool_sinks, 0.022)], ids=["tiny", "verify", "two_pool"])
def test_e4m3_p_alone_moves_the_pages_workloads_past_a_flat_two_percent(make, low):
    """The datapath the Kimi K3.1 attn_sparse page fixes ("Precision": every
    P rounded to E4M3 at 448 of the running maximum, FP32 elsewhere) is, on
    the pages' three small workloads, itself more than 2% of the row maximum
    away from the FP64 definition: rounding P to three mantissa bits moves a
    weight by up to 1/16 of itself. A flat 0.02 * max|row| bound against the
    definition is therefore not met by the pages' own arithmetic; the GPU
    tests bound the distance to the definition by max(0.02 * max|row|, the
    propagated E4M3 error) and hold the GPU to 2e-3 of the emulated datapath.
    The partition (one split, 128-column chunks) does not change this."""
    w = make()
    prob = oracle.Problem.from_workload(w)
    ref, ref_lse = oracle.fp64(prob)
    emu, _, _ = oracle.emulate(prob, 1, 128)
    live = ~np.isneginf(ref_lse)
    rowmax = np.abs(ref[live]).max(axis=1, keepdims=True)
    worst = (np.abs(emu[live] - ref[live]) / rowmax).max()
    assert worst > low, worst
    # and rounding P is the whole of it: without the E4M3 step the emulation
    # is within FP32 roundings of the definition
    plain, _, _ = oracle.emulate(prob, 1, 128, flags=oracle.NO_P_ROUNDING)
    assert (np.abs(plain[live] - ref[live]) / rowmax).max() < 1e-5
