"""Shared helpers of the GPU parity tests: device copies of a workload, the
library call, and the comparison against both oracle modes."""

from __future__ import annotations

import math

import numpy as np
import torch

from oracle import oracle
from sparse_mla_decode_gb300 import smla

# Tolerances.
#  vs the emulated datapath: |gpu - emu| <= 2e-3 * max|emu row| + 1 BF16 ulp
#    (both sides are rounded to BF16 once, so one rounding step of slack is
#    unavoidable);
#  vs the fp64 definition: |gpu - ref| <= max(0.02 * max|ref row|, E_j) + 1 BF16
#    ulp, where E_j = bmm2*k_scale * sum_k w_k |V_kj| / 16 (+ the subnormal
#    term) bounds what rounding P to E4M3 alone can move element j: the Kimi
#    K3.1 attn_sparse page ("Precision") rounds every P to E4M3 (relative error
#    <= 2^-4 for normal values, absolute <= 2^-10 below 2^-6), and on the
#    pages' own random workloads that already moves elements by up to ~3.7% of
#    the row maximum, past a flat 2% -- the emulated datapath, which has no
#    other error source, shows it;
#  vs the emulated datapath, plus for each element the most that P values
#    within a relative 2^-16 of an E4M3 rounding midpoint can move it by taking
#    their other code (the oracle's tie bound): the GPU's FP32 logits and fast
#    exp2 may put such a P on either side of the midpoint;
#  |lse - lse_ref| <= 1e-3 (base 2).
TOL_FP64 = 0.02
TOL_EMU = 2e-3
TOL_LSE = 1e-3


def to_device(w, device="cuda"):
    d = {
        "q": torch.from_numpy(w["q"]).to(device),
        "pools": [torch.from_numpy(p).to(device) for p in w["pools"]],
        "indices": torch.from_numpy(w["indices"]).to(device),
        "lens": torch.from_numpy(w["lens"]).to(device),
        "sinks": None if w["sinks"] is None else torch.from_numpy(w["sinks"]).to(device),
    }
    return d


def run_gpu(w, d=None, stream=None):
    d = d or to_device(w)
    out, lse = smla.decode(d["q"], d["pools"], d["indices"], d["lens"], d["sinks"],
                           w["bmm1_scale"], w["bmm2_scale"], w["k_scale"],
                           pool_split=w.get("pool_split", 0), stream=stream)
    torch.cuda.synchronize()
    bits = smla.smla_device_error()
    assert bits & smla.DEV_TIMEOUT == 0, f"a bounded wait timed out (device error bits {bits})"
    run_gpu.last_error_bits = bits
    return out.float().cpu().numpy(), out.view(torch.int16).cpu().numpy().view(np.uint16), \
        lse.cpu().numpy()


def plan_of(w):
    T, H, D = w["q"].shape
    shape = smla.make_shape(T, H, w["indices"].shape[1], D, len(w["pools"]), w.get("pool_split", 0))
    return smla.smla_plan_for(shape)


def e4m3_p_bound(w, pairs):
    """Per-element bound on the effect of rounding P to E4M3: the attention
    weights of the definition (torch float64 softmax, a library evaluation)
    applied to |V|, times bmm2*k_scale, / 16, plus the subnormal term
    2^-10 / 448 of the largest weight per key."""
    out = np.zeros((len(pairs), 512))
    D = w["q"].shape[2]
    W = w["indices"].shape[1]
    for i, (t, h) in enumerate(pairs):
        n = max(0, min(int(w["lens"][t]), W))
        rows = []
        for c in range(n):
            r = int(w["indices"][t, c])
            pool = 1 if (len(w["pools"]) == 2 and c >= w.get("pool_split", 0)) else 0
            if 0 <= r < w["pools"][pool].shape[0]:
                rows.append(w["pools"][pool][r])
        if not rows:
            continue
        kv = torch.from_numpy(np.stack(rows)).view(torch.float8_e4m3fn).to(torch.float64)
        q = torch.from_numpy(w["q"][t, h].copy()).view(torch.float8_e4m3fn).to(torch.float64)
        s = (kv @ q) * w["bmm1_scale"]
        logits = s
        if w["sinks"] is not None:
            logits = torch.cat([s, torch.tensor([float(w["sinks"][h])], dtype=torch.float64)])
        p = torch.softmax(logits, 0)[: s.shape[0]]
        absv = kv[:, :512].abs()
        a = (p[:, None] * absv).sum(0) / 16.0 + (2.0 ** -10 / 448.0) * absv.sum(0) * p.max()
        out[i] = a.numpy() * w["bmm2_scale"] * w["k_scale"]
    return out


def bf16_ulp(x):
    """Spacing of BF16 numbers at |x| (8 significand bits; FP32's exponent
    range, so 2^-133 throughout the subnormal range below 2^-126)."""
    a = np.abs(np.asarray(x, np.float64))
    a = np.maximum(a, 2.0 ** -126)
    e = np.floor(np.log2(a))
    return 2.0 ** (e - 7)


def compare(w, got, got_bits, got_lse, pairs=None, emulate=True):
    """Checks GPU results (rows in ``pairs`` order, or all (t, h)) against the
    oracle's fp64 definition and its emulated datapath on the GPU's plan."""
    prob = oracle.Problem.from_workload(w)
    T, H = w["q"].shape[:2]
    if pairs is None:
        pairs = [(t, h) for t in range(T) for h in range(H)]
    pairs = np.asarray(pairs, np.int32).reshape(-1, 2)
    g = got.reshape(T, H, -1)[pairs[:, 0], pairs[:, 1]]
    gb = got_bits.reshape(T, H, -1)[pairs[:, 0], pairs[:, 1]]
    gl = got_lse.reshape(T, H)[pairs[:, 0], pairs[:, 1]]
    ref, ref_lse = oracle.fp64(prob, pairs)
    report = {}
    failures = []
    empty = np.isneginf(ref_lse)
    # empty rows: +0.0 bits and -inf, exactly
    if not np.all(gb[empty] == 0):
        failures.append("empty rows must be +0.0")
    if not np.all(np.isneginf(gl[empty])):
        failures.append("empty rows must have lse -inf")
    live = ~empty
    if live.any():
        rowmax = np.abs(ref[live]).max(axis=1, keepdims=True)
        err = np.abs(g[live] - ref[live])
        e4m3 = e4m3_p_bound(w, pairs[live])
        bound = np.maximum(TOL_FP64 * rowmax, e4m3) + bf16_ulp(ref[live])
        worst = (err / bound).max()
        report["fp64_worst_frac_of_bound"] = round(float(worst), 4)
        report["fp64_max_rel_err"] = round(float((err / rowmax).max()), 5)
        report["fp64_frac_of_flat_2pct"] = round(float((err / (TOL_FP64 * rowmax + bf16_ulp(ref[live]))).max()), 4)
        if worst > 1.0:
            failures.append(f"fp64 parity: worst error at {worst:.3f} of the bound")
        lerr = np.abs(gl[live] - ref_lse[live])
        report["lse_max_abs_err"] = float(lerr.max())
        if lerr.max() > TOL_LSE:
            failures.append(f"lse error {lerr.max()}")
    if emulate:
        plan = plan_of(w)
        val, bits, emu_lse, ties = oracle.emulate(prob, plan["splits"], plan["chunk"], pairs, ties=True)
        if not np.array_equal(np.isneginf(emu_lse), empty):
            failures.append("emulated empty rows differ")
        if live.any():
            rowmax = np.abs(val[live]).max(axis=1, keepdims=True)
            err = np.abs(g[live] - val[live])
            bound = TOL_EMU * rowmax + bf16_ulp(val[live]) + ties[live]
            worst = (err / bound).max()
            report["emu_worst_frac_of_bound"] = round(float(worst), 4)
            report["emu_max_rel_err"] = round(float((err / rowmax).max()), 6)
            report["emu_bits_equal_frac"] = round(float(np.mean(gb[live] == bits[live])), 5)
            lerr = np.abs(gl[live] - emu_lse[live]).max()
            report["emu_lse_max_abs_err"] = float(lerr)
            if worst > 1.0:
                failures.append(f"emulated parity: worst error at {worst:.3f} of the bound")
            if lerr > TOL_LSE:
                failures.append(f"emulated lse error {lerr}")
    print("parity", w.get("name"), report)
    assert not failures, "; ".join(failures) + f" {report}"
    return report


def log2e():
    return 1.0 / math.log(2.0)
