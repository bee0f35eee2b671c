"""Host-side accounting of bench.py: algorithmic bytes per call, the source
hashes that tie a committed DRAM-traffic figure to the kernel it was taken on,
and the lookup that reports it. No GPU."""

import json
import os

import pytest
import torch

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_merge_bytes_live_counts_only_rows_with_weight():
    S, T, H = 3, 4, 2
    lses = torch.zeros((S, T, H))
    lens = torch.full((T,), 5, dtype=torch.int32)
    full = bench.merge_bytes_live(lses, lens)
    assert full == bench.merge_bytes(S, T, H)  # every row live: the upper bound
    lses[0, 1, 1] = float("-inf")
    lses[2, 3, 0] = float("nan")
    assert bench.merge_bytes_live(lses, lens) == full - 2 * 1024
    lens[2] = 0  # a token without keys: none of its S * H rows is read
    assert bench.merge_bytes_live(lses, lens) == full - 2 * 1024 - S * H * 1024


def test_merge_value_bytes_live_adds_the_projection_operands():
    S, T, H = 2, 3, 4
    lses = torch.zeros((S, T, H))
    lens = torch.full((T,), 1, dtype=torch.int32)
    assert bench.merge_value_bytes_live(lses, lens) == bench.merge_value_bytes(S, T, H)
    lses[1, 0, 2] = float("-inf")
    assert bench.merge_value_bytes_live(lses, lens) == bench.merge_value_bytes(S, T, H) - 1024


def test_value_bytes_formula():
    T, H = 64, 128
    # merged rows, W_UV, gates in, values out, counts
    assert bench.value_bytes(T, H) == T * H * 1024 + H * 512 * 128 * 2 + 2 * T * H * 256 + 4 * T


@pytest.mark.parametrize("config", ["batch", "value", "merge_value", "merge", "mxfp4"])
def test_kernel_sha_is_stable_and_tracks_the_sources(config):
    a, b = bench.kernel_sha(config), bench.kernel_sha(config)
    assert a == b and len(a) == 16
    names = bench.KERNEL_SOURCES.get(config, ("smla_decode.cu", "smla_ptx.cuh"))
    for n in names:
        assert os.path.exists(os.path.join(ROOT, "sparse_mla_decode_gb300", "csrc", n))


def test_configs_with_distinct_kernels_hash_differently():
    shas = {c: bench.kernel_sha(c) for c in ("batch", "value", "merge", "mxfp4")}
    assert len(set(shas.values())) == 4


def test_traffic_is_reported_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        recorded = json.load(f)
    for config, entry in recorded.items():
        expected = entry["dram_bytes_per_launch"] if entry["kernel_sha"] == bench.kernel_sha(config) else None
        assert bench.ncu_traffic(config) == expected
    # a record taken on another source is not reported
    fake_root = tmp_path
    (fake_root / "profiles").mkdir()
    stale = {"batch": dict(recorded.get("batch", {}), kernel_sha="0" * 16, dram_bytes_per_launch=1)}
    (fake_root / "profiles" / "dram_traffic.json").write_text(json.dumps(stale))
    real = {c: bench.kernel_sha(c) for c in ("batch", "value")}
    monkeypatch.setattr(bench, "kernel_sha", lambda config="batch": real[config])
    monkeypatch.setattr(bench, "ROOT", str(fake_root))
    assert bench.ncu_traffic("batch") is None
    assert bench.ncu_traffic("value") is None  # no record at all


def test_fp8_peak_is_the_committed_microbenchmark_figure():
    peak, source = bench.fp8_peak()
    with open(os.path.join(ROOT, "profiles", "fp8_mma_peak.json")) as f:
        assert peak == json.load(f)["fp8_dense_peak_tflops"]
    assert "measured" in source and "tcgen05" in source


def test_ds_mla_bytes_counts_656_byte_rows_q_and_out():
    from sparse_mla_decode_gb300 import workloads

    w = workloads.ds_mla_small("acct", seed=1, tokens=2, heads=32, width=40, pool_rows=100, holes=0.2)
    rows = workloads.unique_active_rows(w)
    assert bench.ds_mla_bytes(w) == rows * 656 + 2 * 32 * (512 + 128) + 2 * 32 * 512 * 2


def test_cpu_baseline_times_all_cores_and_one_core_as_medians_of_three():
    from sparse_mla_decode_gb300 import workloads

    cpu = bench.cpu_oracle_rate([workloads.tiny()], 0.3)
    assert cpu["kind"] == "oracle" and cpu["unit"] == "GB/s" and cpu["value"] > 0
    assert cpu["one_core"]["cores"] == 1 and cpu["one_core"]["value"] > 0
    assert "median of 3" in cpu["sample"] and "median of 3" in cpu["one_core"]["sample"]


def test_reference_arm_reports_its_measured_step_and_whether_it_extrapolates():
    import subprocess
    import sys

    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "2", "--warmup", "0"], capture_output=True, text=True, check=True, cwd=ROOT)
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["extrapolated"] is False  # 16 pairs: the whole call per step
    assert line["ms_per_step"] * 1e3 == pytest.approx(line["us_per_call_extrapolated"], rel=1e-3)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_gather_floor_counts_shared_rows_at_the_hot_rate():
    import numpy as np

    with open(os.path.join(ROOT, "profiles", "row_gather_peak.json")) as f:
        rates = {(r["method"], r["issuers"], r["pool"]): r["sm_bytes_per_ns"] for r in json.load(f)["rows"]}
    # two tokens of 8 columns: rows 0-3 shared by both (hot), 4 more each of their own (cold), one hole
    idx = np.array([[0, 1, 2, 3, 10, 11, 12, 13], [0, 1, 2, 3, 20, 21, 22, -1]], np.int32)
    w = {"q": np.zeros((2, 16, 576), np.uint8), "indices": idx, "lens": np.array([8, 8], np.int32)}
    plan = {"pair": 1, "splits": 1, "chunks_per_split": 1, "chunk": 128, "ctas": 2, "resident_ctas": 152}
    want = (4 * 576 / rates[(0, 7, "hot")] + 4 * 576 / rates[(0, 7, "cold")]) / 1e3  # token 0, the slower
    got = bench.gather_floor(w, plan)
    assert got["us"] == pytest.approx(want, abs=0.01) and got["method"] == "cp.async"
    plan["pair"] = 2
    assert bench.gather_floor(w, plan)["method"] == "paired tile::gather4 multicast"


def test_kernel_hash_sees_code_not_comments():
    """The committed DRAM traffic is keyed by the kernel's code: editing a
    comment or the layout keeps the key, changing an expression or a string
    literal does not."""
    base = 'int f(int x) { return x + 1; }  // one\n/* note */ const char* s = "a // b";\n'
    assert bench.code_text(base) == bench.code_text(
        'int f(int x)   {\n  return x + 1;\n}  // another note\nconst char* s = "a // b"; /* x */\n')
    assert bench.code_text(base) != bench.code_text(base.replace("x + 1", "x + 2"))
    assert bench.code_text(base) != bench.code_text(base.replace('"a // b"', '"a // c"'))
    assert bench.code_text('char c = \'/\'; // q') == "char c = '/';"
