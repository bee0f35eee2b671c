"""GPU parity: libsmla.so (through its C ABI) against both oracle modes.

Sizes run from the three small workloads of the pages (1 x 16 heads x 256
keys; 5 verify rows x 128 heads with an empty row; 12 tokens x 16 heads over
two pools with sinks) through ragged and degenerate cases to the full
64 x 128 x 2048 batch, sampled per (token, head)."""

import os

import numpy as np
import pytest
import torch

from sparse_mla_decode_gb300 import smla, workloads
from tests.gpu_helpers import compare, plan_of, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture
def forced_splits():
    old = os.environ.get("SMLA_SPLITS")

    def set_splits(s):
        if s is None:
            os.environ.pop("SMLA_SPLITS", None)
        else:
            os.environ["SMLA_SPLITS"] = str(s)

    yield set_splits
    set_splits(old)


def test_library_loads_and_reports_version():
    assert smla.smla_version() == 200
    assert smla.smla_device_error() == 0


@pytest.mark.parametrize("make", [workloads.tiny, workloads.verify_rows, workloads.two_pool_sinks],
                         ids=["tiny", "verify", "two_pool"])
def test_page_workloads(make):
    w = make()
    got, bits, lse = run_gpu(w)
    report = compare(w, got, bits, lse)
    print(w["name"], plan_of(w), report)
    assert smla.smla_device_error() == 0


SMALL = [
    # heads, head_dim, width, holes, sinks, lens (None = full)
    (16, 576, 300, 0.0, False, None),
    (16, 512, 130, 0.1, True, None),
    (32, 576, 257, 0.05, False, None),
    (48, 576, 200, 0.0, True, None),
    (64, 576, 384, 0.1, True, [384, 1, 129]),
    (64, 512, 250, 0.0, False, [250, 0, 77]),
    (128, 576, 129, 0.2, False, None),
    (80, 512, 600, 0.02, True, None),
]


@pytest.mark.parametrize("case", SMALL, ids=[f"h{c[0]}_d{c[1]}_w{c[2]}" for c in SMALL])
def test_small_shapes(case):
    heads, dim, width, holes, sinks, lens = case
    tokens = 3 if lens is not None else 2
    w = workloads.small("small", seed=heads * 1000 + width, tokens=tokens, heads=heads, width=width,
                        head_dim=dim, pool_rows=4096, holes=holes, sinks=sinks, lens=lens)
    got, bits, lse = run_gpu(w)
    print(case, plan_of(w), compare(w, got, bits, lse))


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 5, 8, 16])
def test_forced_split_counts(forced_splits, splits):
    forced_splits(splits)
    w = workloads.small("splits", seed=77, tokens=2, heads=64, width=2048, head_dim=576,
                        pool_rows=8192, holes=0.05, sinks=True, lens=[2048, 1000])
    plan = plan_of(w)
    chunks = plan["chunks"]
    per = -(-chunks // splits)
    assert plan["splits"] == -(-chunks // per)  # no split without chunks at full width
    got, bits, lse = run_gpu(w)
    print(splits, plan, compare(w, got, bits, lse))


@pytest.fixture
def env():
    saved = {}

    def set_env(name, value):
        if name not in saved:
            saved[name] = os.environ.get(name)
        if value is None:
            os.environ.pop(name, None)
        else:
            os.environ[name] = str(value)

    yield set_env
    for name, value in saved.items():
        if value is None:
            os.environ.pop(name, None)
        else:
            os.environ[name] = value


PAIRED = [
    # heads, head_dim, width, forced head tile, forced splits, lens
    (128, 576, 2048, None, None, [2048, 1000, 5]),
    (128, 576, 700, None, 3, [700, 699, 300]),
    (64, 512, 1300, 16, 2, [1300, 640, 641]),
    (32, 576, 257, 16, 1, [257, 0, 128]),
    (128, 576, 900, 32, 8, [900, 129, 850]),
]


@pytest.mark.parametrize("case", PAIRED, ids=[f"h{c[0]}_d{c[1]}_w{c[2]}_t{c[3]}_s{c[4]}" for c in PAIRED])
def test_paired_head_groups(env, case):
    """Head-group pairs sharing each chunk's gather (tile::gather4 multicast),
    with and without split merges across the pair's cluster."""
    heads, dim, width, tile, splits, lens = case
    env("SMLA_PAIR", 1)
    env("SMLA_HEAD_TILE", tile)
    env("SMLA_SPLITS", splits)
    w = workloads.small("paired", seed=heads + width, tokens=3, heads=heads, width=width, head_dim=dim,
                        pool_rows=6000, holes=0.07, sinks=True, lens=lens)
    plan = plan_of(w)
    assert plan["pair"] == 2
    got, bits, lse = run_gpu(w)
    print(case, plan, compare(w, got, bits, lse))


CHUNK96 = [
    # tokens, heads, head_dim, width, forced head tile, forced splits, pair, lens
    (3, 64, 576, 300, 64, None, 0, [300, 97, 0]),      # ragged tail: 96 + 96 + 96 + 12
    (2, 64, 512, 2048, 32, None, 0, [2048, 1111]),
    (3, 128, 576, 1000, 64, None, 1, [1000, 96, 950]),  # paired, gather4 multicast
    (4, 64, 576, 2048, 64, 3, 0, [2048, 2000, 1500, 193]),  # split merge over three CTAs
    (2, 128, 576, 777, 64, 2, 1, [777, 500]),          # paired and split
]


@pytest.mark.parametrize("case", CHUNK96, ids=[f"t{c[0]}_h{c[1]}_d{c[2]}_w{c[3]}_s{c[5]}_p{c[6]}" for c in CHUNK96])
def test_chunks_of_96_keys_in_three_stages(env, case):
    """The three-stage pipeline of 96-key chunks (the MMAs read 128 rows; the
    32 past each chunk are masked in S^T and never read by PV)."""
    tokens, heads, dim, width, tile, splits, pair, lens = case
    env("SMLA_CHUNK", 96)
    env("SMLA_HEAD_TILE", tile)
    env("SMLA_SPLITS", splits)
    env("SMLA_PAIR", pair)
    w = workloads.small("chunk96", seed=tokens * 1000 + width, tokens=tokens, heads=heads, width=width,
                        head_dim=dim, pool_rows=5000, holes=0.08, sinks=True, lens=lens)
    plan = plan_of(w)
    assert plan["chunk"] == 96 and plan["pair"] == (2 if pair else 1), plan
    got, bits, lse = run_gpu(w)
    print(case, plan, compare(w, got, bits, lse))


PAIR_KERNEL = [
    # tokens, heads, head_dim, width, lens, holes, sinks, two pools (split column)
    (3, 128, 576, 2048, [2048, 1000, 5], 0.07, True, None),
    (3, 128, 576, 700, [700, 699, 300], 0.0, False, None),
    (3, 128, 512, 1300, [1300, 640, 641], 0.07, True, None),
    (3, 256, 576, 257, [257, 0, 128], 0.05, True, None),
    (4, 128, 512, 640, [640, 300, 129, 0], 0.05, True, 128),
    (2, 128, 576, 256, [256, 255], 0.0, False, None),
]


@pytest.mark.parametrize("case", PAIR_KERNEL,
                         ids=[f"t{c[0]}_h{c[1]}_d{c[2]}_w{c[3]}{'_pools' if c[7] else ''}" for c in PAIR_KERNEL])
def test_pair_kernel(env, case):
    """The 128-head CTA-pair kernel (cta_group::2 products, the softmax over
    256-key chunks split across the pair) on ragged counts, holes, sinks, two
    pools, 512-byte rows, two head groups and an empty token."""
    tokens, heads, dim, width, lens, holes, sinks, split = case
    env("SMLA_KERNEL", "pair")
    w = workloads.small("pair", seed=heads + width + tokens, tokens=tokens, heads=heads, width=width,
                        head_dim=dim, pool_rows=6000, holes=holes, sinks=sinks, lens=lens,
                        two_pools=split is not None, pool_split=split or 0)
    plan = plan_of(w)
    assert (plan["pair"], plan["head_tile"], plan["chunk"], plan["splits"]) == (2, 128, 256, 1)
    got, bits, lse = run_gpu(w)
    print(case, plan, compare(w, got, bits, lse))


@pytest.mark.parametrize("kernel", ["tile", "pair"])
def test_128_heads_both_kernels(env, kernel):
    """The same 128-head workload through either kernel, each against the
    oracle's emulation of its own partition (128- or 256-column chunks)."""
    env("SMLA_KERNEL", kernel)
    w = workloads.small("both", seed=404, tokens=5, heads=128, width=600, head_dim=576, pool_rows=8192,
                        holes=0.1, sinks=True, lens=[600, 599, 1, 256, 300])
    got, bits, lse = run_gpu(w)
    print(kernel, plan_of(w), compare(w, got, bits, lse))


# Launches of more CTAs than the GPU holds at once (several waves), sampled
# against both oracle modes: the sweep's 256-token points at 128 and 16 heads,
# and its recipe of 10% holes with counts uniform in [k/2, k].
MULTI_WAVE = [
    # tokens, heads, width, holes, counts in [k/2, k]
    (256, 128, 2048, 0.0, False),
    (256, 16, 256, 0.0, False),
    (128, 64, 1024, 0.1, True),
]


@pytest.mark.parametrize("case", MULTI_WAVE, ids=[f"t{c[0]}_h{c[1]}_k{c[2]}" for c in MULTI_WAVE])
def test_multi_wave_launches_sampled(case):
    tokens, heads, width, holes, ragged = case
    w = workloads.sweep_point(tokens, heads, width, seed=tokens * 7 + heads + width, pool_rows=1 << 18) if ragged else \
        workloads.small("waves", seed=tokens + heads + width, tokens=tokens, heads=heads, width=width, head_dim=576,
                        pool_rows=1 << 18, holes=holes)
    plan = plan_of(w)
    got, bits, lse = run_gpu(w)
    rng = np.random.default_rng(tokens + heads)
    pairs = np.stack([rng.integers(0, tokens, 64), rng.integers(0, heads, 64)], axis=1)
    print(case, plan, compare(w, got, bits, lse, pairs=pairs))


def test_two_pools_ragged_split_boundary():
    w = workloads.small("pools", seed=91, tokens=4, heads=16, width=333, head_dim=512,
                        pool_rows=1000, two_pools=True, pool_split=77, holes=0.05, sinks=True,
                        lens=[333, 76, 78, 200])
    got, bits, lse = run_gpu(w)
    print(compare(w, got, bits, lse))


def test_degenerate_inputs():
    w = workloads.small("degenerate", seed=5, tokens=6, heads=16, width=140, head_dim=576,
                        pool_rows=512, lens=[0, -3, 500, 140, 1, 129], sinks=True)
    w["indices"][3, :] = -1  # every column a hole
    got, bits, lse = run_gpu(w)
    compare(w, got, bits, lse)
    assert np.all(bits[[0, 1, 3]] == 0) and np.all(np.isneginf(lse[[0, 1, 3]]))


def test_zero_width_and_zero_tokens():
    w = workloads.small("zero", seed=6, tokens=2, heads=16, width=0, head_dim=576)
    got, bits, lse = run_gpu(w)
    assert np.all(bits == 0) and np.all(np.isneginf(lse))
    d = to_device(w)
    q = d["q"][:0]
    out = torch.empty((0, 16, 512), dtype=torch.bfloat16, device="cuda")
    smla.smla_decode(q, d["pools"], d["indices"][:0], d["lens"][:0], None, 1.0, 1.0, 1.0, out, None)


def test_index_beyond_pool_is_masked_and_flagged():
    w = workloads.small("oob", seed=7, tokens=1, heads=16, width=64, head_dim=576, pool_rows=100)
    w["indices"][0, 10] = 100  # one past the last row
    w["indices"][0, 11] = 2 ** 30
    got, bits, lse = run_gpu(w)
    assert run_gpu.last_error_bits == smla.DEV_INDEX_RANGE
    compare(w, got, bits, lse)  # the oracle treats them as holes too
    assert smla.smla_device_error() == 0


def test_strided_layouts_match_contiguous():
    w = workloads.small("strided", seed=8, tokens=3, heads=32, width=200, head_dim=576,
                        pool_rows=2048, holes=0.1, sinks=True)
    d = to_device(w)
    out0, lse0 = smla.decode(d["q"], d["pools"], d["indices"], d["lens"], d["sinks"],
                             w["bmm1_scale"], w["bmm2_scale"], w["k_scale"])
    T, H, D = w["q"].shape
    qbig = torch.zeros((T, H + 16, D + 64), dtype=torch.uint8, device="cuda")
    qbig[:, 8:8 + H, :D] = d["q"]
    q = qbig[:, 8:8 + H, :D]
    ibig = torch.full((T, 256), -1, dtype=torch.int32, device="cuda")
    ibig[:, :200] = d["indices"]
    obig = torch.zeros((T, H + 3, 640), dtype=torch.bfloat16, device="cuda")
    out = obig[:, 1:1 + H, :512]
    lbig = torch.zeros((T, 40), dtype=torch.float32, device="cuda")
    lse = lbig[:, :H]
    smla.smla_decode(q, d["pools"], ibig[:, :200], d["lens"], d["sinks"], w["bmm1_scale"],
                     w["bmm2_scale"], w["k_scale"], out, lse)
    torch.cuda.synchronize()
    assert smla.smla_device_error() == 0
    assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
    assert torch.equal(lse, lse0)
    assert torch.all(obig[:, 0] == 0) and torch.all(obig[:, :, 512:] == 0)


def test_repeated_calls_are_bitwise_deterministic():
    w = workloads.small("det", seed=9, tokens=4, heads=64, width=700, head_dim=576,
                        pool_rows=4096, holes=0.05)
    d = to_device(w)
    a = smla.decode(d["q"], d["pools"], d["indices"], d["lens"], None, w["bmm1_scale"], 1.0, 1.0)
    b = smla.decode(d["q"], d["pools"], d["indices"], d["lens"], None, w["bmm1_scale"], 1.0, 1.0)
    torch.cuda.synchronize()
    assert smla.smla_device_error() == 0
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])


def test_bandwidth_batch_full_size_sampled():
    """64 tokens x 128 heads x 2048 keys on the 1M-row pool, in the launch
    configuration the benchmark times; 96 (token, head) pairs against the
    oracle, every LSE finite."""
    w = workloads.bandwidth_batch()
    got, bits, lse = run_gpu(w)
    rng = np.random.default_rng(1)
    pairs = np.stack([rng.integers(0, 64, 96), rng.integers(0, 128, 96)], axis=1)
    print(plan_of(w), compare(w, got, bits, lse, pairs=pairs))
    assert np.all(np.isfinite(lse))


def test_back_to_back_calls_with_dependent_launch():
    """Many calls in a row on one stream (programmatic dependent launch lets
    each start before the previous ends) over rotating inputs: no bounded wait
    may time out and every result must equal its single-call result."""
    sets = [workloads.small("b2b", seed=100 + r, tokens=8, heads=128, width=2048, head_dim=576,
                            pool_rows=1 << 15, holes=0.02) for r in range(3)]
    devs = [to_device(w) for w in sets]
    ref = []
    for w, d in zip(sets, devs):
        o, l = smla.decode(d["q"], d["pools"], d["indices"], d["lens"], None, w["bmm1_scale"], 1.0, 1.0)
        torch.cuda.synchronize()
        ref.append((o.clone(), l.clone()))
    outs = [smla.decode(devs[i % 3]["q"], devs[i % 3]["pools"], devs[i % 3]["indices"],
                        devs[i % 3]["lens"], None, sets[i % 3]["bmm1_scale"], 1.0, 1.0)
            for i in range(60)]
    torch.cuda.synchronize()
    assert smla.smla_device_error() == 0
    for i, (o, l) in enumerate(outs):
        assert torch.equal(o.view(torch.int16), ref[i % 3][0].view(torch.int16))
        assert torch.equal(l, ref[i % 3][1])
