"""The seeded input generators follow the recipes the design states for each
workload: shapes, index structure (unique rows, holes, counts, pools, the
shared hot set), value distributions and the fp8_ds_mla row packing. CPU only;
the large pools are drawn smaller here, with the same recipe."""

import inspect
import math

import numpy as np
import pytest
import torch

from sparse_mla_decode_gb300 import workloads


def e4m3_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_normal_codes_are_finite_standard_normals():
    codes = workloads.e4m3_normal(np.random.default_rng(0), (200_000,))
    assert codes.dtype == np.uint8
    assert not np.any((codes & 0x7F) == 0x7F), "no NaN codes"
    x = e4m3_values(codes)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.02


def test_tiny():
    w = workloads.tiny()
    assert w["q"].shape == (1, 16, 576) and w["pools"][0].shape == (4096, 576)
    idx = w["indices"][0]
    assert idx.shape == (256,) and np.unique(idx).size == 256 and idx.min() >= 0 and idx.max() < 4096
    assert int(w["lens"][0]) == 256 and w["sinks"] is None
    assert w["bmm1_scale"] == pytest.approx(1 / math.sqrt(192))


def test_verify_rows():
    w = workloads.verify_rows()
    assert w["q"].shape == (5, 128, 576) and w["pools"][0].shape == (65536, 576)
    assert w["k_scale"] == 0.05 and int(w["lens"][2]) == 0
    for t in range(5):
        n = int(w["lens"][t])
        assert n == 0 or 64 <= n <= 256
        row = w["indices"][t]
        assert np.all(row[n:] == -1)
        assert np.unique(row[:n]).size == n and (n == 0 or (row[:n].min() >= 0 and row[:n].max() < 65536))


def test_two_pool_sinks():
    w = workloads.two_pool_sinks()
    assert w["q"].shape == (12, 16, 512)
    assert [p.shape for p in w["pools"]] == [(8192, 512), (262144, 512)] and w["pool_split"] == 128
    idx = w["indices"]
    live = idx >= 0
    assert np.all(idx[:, :128][live[:, :128]] < 8192) and np.all(idx[:, 128:][live[:, 128:]] < 262144)
    assert 0.03 < (~live).mean() < 0.07  # 5 % holes
    assert np.all((w["lens"] >= 300) & (w["lens"] <= 640))
    assert w["sinks"].shape == (16,) and w["bmm2_scale"] == 0.5
    assert w["bmm1_scale"] == pytest.approx(1 / math.sqrt(512))


@pytest.mark.parametrize("make", [workloads.bandwidth_batch, workloads.ds_mla_batch])
def test_batch_index_recipe_half_from_a_shared_hot_set(make):
    sig = inspect.signature(make).parameters
    assert sig["tokens"].default == 64 and sig["heads"].default == 128 and sig["topk"].default == 2048
    assert sig["pool_rows"].default == 1 << 20 and sig["hot_rows"].default == 20000
    pool_rows, hot_rows, W = 1 << 14, 1000, 256
    w = make(tokens=6, heads=16, topk=W, pool_rows=pool_rows, hot_rows=hot_rows)
    idx = w["indices"]
    assert np.all(w["lens"] == W) and w["sinks"] is None
    counts = {}
    for t in range(6):
        assert np.unique(idx[t]).size == W and idx[t].min() >= 0 and idx[t].max() < pool_rows
        for r in idx[t]:
            counts[int(r)] = counts.get(int(r), 0) + 1
    # the hot set: every row shared by two tokens or more comes from it, and
    # each token draws exactly half of its rows there
    shared = {r for r, n in counts.items() if n > 1}
    assert len(shared) <= hot_rows
    for t in range(6):
        in_shared = sum(1 for r in idx[t] if int(r) in shared)
        assert in_shared <= W // 2
    rng_rows = np.concatenate([idx[t] for t in range(6)])
    assert np.unique(rng_rows).size < 6 * W  # tokens overlap


def test_sweep_point():
    w = workloads.sweep_point(4, 16, 256, pool_rows=1 << 12)
    idx = w["indices"]
    assert w["q"].shape == (4, 16, 576) and idx.shape == (4, 256)
    assert 0.05 < (idx < 0).mean() < 0.16  # 10 % holes
    assert np.all((w["lens"] >= 128) & (w["lens"] <= 256))
    for t in range(4):
        live = idx[t][idx[t] >= 0]
        assert np.unique(live).size == live.size


def test_ds_mla_rows_pack_codes_scales_and_rope():
    rows = workloads.ds_mla_rows(np.random.default_rng(3), 20000)
    assert rows.shape == (20000, workloads.DS_MLA_ROW) == (20000, 656) and rows.dtype == np.uint8
    codes = rows[:, :512]
    assert not np.any((codes & 0x7F) == 0x7F)
    scales = rows[:, 512:528].copy().view("<f4").astype(np.float64)
    mant, expo = np.frexp(scales)  # scale = mant * 2^expo, mant in [0.5, 1)
    assert np.all((mant >= 0.5) & (mant < 1.0))
    assert set(np.unique(expo).tolist()) == set(range(-6, 3))  # u uniform over -6..2
    rope = torch.from_numpy(rows[:, 528:].copy().view("<i2")).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.all(np.isfinite(rope)) and abs(rope.std() - 1.0) < 0.02


def test_merge_sets():
    parts, lses, lens = workloads.merge_sets(sources=4, tokens=8, heads=16)
    assert parts.shape == (4, 8, 16, 512) and parts.dtype == torch.bfloat16
    empty = torch.isneginf(lses)
    live = lses[~empty]
    assert bool(((live >= 4) & (live < 12)).all())
    assert 0.005 < empty.float().mean().item() < 0.08  # 3 % empty sources
    assert int(lens[5]) == 0 and int(lens[0]) == 2048
