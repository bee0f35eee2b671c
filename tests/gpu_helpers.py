"""Shared helpers of the GPU parity tests: device copies of a workload, the
library call, and the comparison against both oracle modes."""

from __future__ import annotations

import math

import numpy as np
import torch

from oracle import oracle
from sparse_mla_decode_gb300 import smla

# Spec tolerances: |gpu - fp64| <= 0.02 * max|ref row| + 1 BF16 ulp;
# |gpu - emulated| <= 2e-3 * max|emulated row| + 1 BF16 ulp (both sides are
# rounded to BF16 once, so one rounding step of slack is unavoidable);
# |lse - lse_ref| <= 1e-3 (base 2).
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
    return out.float().cpu().numpy(), out.view(torch.int16).cpu().numpy().view(np.uint16), \
        lse.cpu().numpy()


def plan_of(w):
    T, H, D = w["q"].shape
    shape = smla.make_shape(T, H, w["indices"].shape[1], D, len(w["pools"]), w.get("pool_split", 0))
    return smla.smla_plan_for(shape)


def bf16_ulp(x):
    a = np.abs(np.asarray(x, np.float64))
    a = np.maximum(a, 2.0 ** -133)
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
    empty = np.isneginf(ref_lse)
    # empty rows: +0.0 bits and -inf, exactly
    assert np.all(gb[empty] == 0), "empty rows must be +0.0"
    assert np.all(np.isneginf(gl[empty])), "empty rows must have lse -inf"
    live = ~empty
    if live.any():
        rowmax = np.abs(ref[live]).max(axis=1, keepdims=True)
        err = np.abs(g[live] - ref[live])
        bound = TOL_FP64 * rowmax + bf16_ulp(ref[live])
        worst = (err / bound).max()
        report["fp64_worst_frac_of_bound"] = float(worst)
        report["fp64_max_rel_err"] = float((err / rowmax).max())
        assert worst <= 1.0, f"fp64 parity: worst error at {worst:.3f} of the bound"
        lerr = np.abs(gl[live] - ref_lse[live])
        report["lse_max_abs_err"] = float(lerr.max())
        assert lerr.max() <= TOL_LSE, f"lse error {lerr.max()}"
    if emulate:
        plan = plan_of(w)
        val, bits, emu_lse = oracle.emulate(prob, plan["splits"], plan["chunk"], pairs)
        assert np.array_equal(np.isneginf(emu_lse), empty)
        if live.any():
            rowmax = np.abs(val[live]).max(axis=1, keepdims=True)
            err = np.abs(g[live] - val[live])
            bound = TOL_EMU * rowmax + bf16_ulp(val[live])
            worst = (err / bound).max()
            report["emu_worst_frac_of_bound"] = float(worst)
            report["emu_max_rel_err"] = float((err / rowmax).max())
            report["emu_bits_equal_frac"] = float(np.mean(gb[live] == bits[live]))
            assert worst <= 1.0, f"emulated parity: worst error at {worst:.3f} of the bound"
            assert np.abs(gl[live] - emu_lse[live]).max() <= TOL_LSE
    return report


def log2e():
    return 1.0 / math.log(2.0)
