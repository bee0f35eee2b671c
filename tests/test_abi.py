"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every function include/smla.h declares, plans
launches, and rejects bad arguments before launching anything."""

import ctypes
import os
import re

import pytest

from sparse_mla_decode_gb300 import build, smla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return smla.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "smla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(smla_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "smla_decode" in names and "smla_plan_for" in names
    for name in names:
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def shape(**kw):
    base = dict(tokens=64, heads=128, width=2048, head_dim=576)
    base.update(kw)
    return smla.make_shape(**base)


def test_plan_bandwidth_batch(lib):
    p = smla.smla_plan_for(shape(), num_sms=152)
    assert p["head_tile"] == 64 and p["head_groups"] == 2 and p["chunk"] == 96 and p["pair"] == 2
    assert p["chunks"] == 22 and p["splits"] * p["chunks_per_split"] >= 22
    assert p["ctas"] == 64 * 2 * p["splits"]
    assert p["smem_bytes"] <= 232448 and p["tmem_columns"] == 512


@pytest.mark.parametrize("tokens,heads,width,chunk,chunks,pair", [
    (128, 64, 2048, 96, 22, 1),   # unpaired, 16 chunks of 128 per CTA: three stages of 96
    (256, 64, 1024, 96, 11, 1),   # unpaired, 8 chunks of 128 per CTA
    (64, 128, 2048, 96, 22, 2),   # paired, 16 chunks of 128 per CTA: three stages of 96
    (64, 128, 1024, 128, 8, 2),   # paired, 8 chunks of 128 per CTA keep two stages of 128
    (32, 64, 2048, 128, 16, 1),   # split four ways: 4 chunks per CTA
    (12, 16, 2048, 128, 16, 1),   # 16-head tiles have no room for a third stage
])
def test_plan_chunk_keys(lib, tokens, heads, width, chunk, chunks, pair):
    p = smla.smla_plan_for(shape(tokens=tokens, heads=heads, width=width), num_sms=152)
    assert (p["chunk"], p["chunks"], p["pair"]) == (chunk, chunks, pair), p
    if chunk == 96:
        assert p["smem_bytes"] > smla.smla_plan_for(shape(tokens=tokens, heads=heads, width=width, head_dim=512),
                                                    num_sms=152)["smem_bytes"]


def test_forced_chunk_keys(lib, monkeypatch):
    monkeypatch.setenv("SMLA_CHUNK", "128")
    assert smla.smla_plan_for(shape(tokens=128, heads=64), num_sms=152)["chunk"] == 128
    monkeypatch.setenv("SMLA_CHUNK", "96")
    p = smla.smla_plan_for(shape(tokens=32, heads=64), num_sms=152)
    assert p["chunk"] == 96 and p["chunks"] == 22 and p["smem_bytes"] <= 232448
    assert smla.smla_plan_for(shape(tokens=64, heads=128), num_sms=152)["chunk"] == 96  # paired, forced
    monkeypatch.setenv("SMLA_HEAD_TILE", "16")
    assert smla.smla_plan_for(shape(tokens=4, heads=64), num_sms=152)["chunk"] == 128


@pytest.mark.parametrize("tokens,heads,width,dim,groups,chunks", [(64, 128, 2048, 576, 1, 8), (5, 256, 256, 576, 2, 1),
                                                                   (12, 128, 640, 512, 1, 3), (256, 128, 2048, 576, 1, 8)])
def test_plan_pair_kernel(lib, monkeypatch, tokens, heads, width, dim, groups, chunks):
    monkeypatch.setenv("SMLA_KERNEL", "pair")
    p = smla.smla_plan_for(shape(tokens=tokens, heads=heads, width=width, head_dim=dim), num_sms=152)
    assert (p["head_tile"], p["head_groups"], p["chunk"], p["chunks"], p["splits"]) == (128, groups, 256, chunks, 1)
    assert p["ctas"] == 2 * tokens * groups and p["resident_ctas"] == 152 and p["pair"] == 2
    assert p["threads"] == 512 and p["tmem_columns"] == 512


def test_plan_pair_kernel_needs_128_head_groups(lib, monkeypatch):
    monkeypatch.setenv("SMLA_KERNEL", "pair")
    for heads in (16, 64, 192):
        assert smla.smla_plan_for(shape(heads=heads), num_sms=152)["head_tile"] <= 64
    monkeypatch.setenv("SMLA_HEAD_TILE", "32")  # a forced tile keeps the tile kernel
    assert smla.smla_plan_for(shape(), num_sms=152)["head_tile"] == 32


@pytest.mark.parametrize("tokens,heads,width,dim", [(1, 16, 256, 576), (5, 128, 256, 576),
                                                    (12, 16, 640, 512), (256, 64, 1024, 576)])
def test_plan_fills_the_machine_without_empty_splits(lib, tokens, heads, width, dim):
    p = smla.smla_plan_for(shape(tokens=tokens, heads=heads, width=width, head_dim=dim), num_sms=152)
    assert 1 <= p["splits"] <= 16
    assert (p["splits"] - 1) * p["chunks_per_split"] < p["chunks"]  # the last split has work
    assert heads % p["head_tile"] == 0


@pytest.mark.parametrize("tokens,heads,width,want", [(1, 16, 2048, 8), (1, 128, 256, 2), (64, 128, 2048, 1),
                                                     (128, 128, 2048, 1), (256, 16, 2048, 1), (32, 16, 1024, 4)])
def test_plan_splits_only_while_resident(lib, tokens, heads, width, want):
    p = smla.smla_plan_for(shape(tokens=tokens, heads=heads, width=width), num_sms=152)
    assert p["splits"] == want
    assert p["resident_ctas"] == (152 // p["splits"]) * p["splits"]
    assert p["splits"] == 1 or p["ctas"] <= p["resident_ctas"]


@pytest.mark.parametrize("tokens,heads,width,tile,splits", [(1, 128, 256, 16, 2), (64, 128, 2048, 64, 1),
                                                            (32, 128, 256, 32, 1), (256, 64, 1024, 64, 1)])
def test_plan_head_tile(lib, tokens, heads, width, tile, splits):
    p = smla.smla_plan_for(shape(tokens=tokens, heads=heads, width=width), num_sms=152)
    assert (p["head_tile"], p["splits"]) == (tile, splits)
    assert p["head_groups"] * p["head_tile"] == heads


@pytest.mark.parametrize("heads,pools,pair", [(128, 1, 2), (64, 1, 1), (128, 2, 1), (16, 1, 1), (32, 1, 1)])
def test_plan_pairs_head_groups(lib, heads, pools, pair):
    kw = dict(tokens=64, heads=heads, width=2048)
    p = smla.smla_plan_for(smla.make_shape(kw["tokens"], heads, kw["width"], 576, pools, 1024 if pools == 2 else 0),
                           num_sms=152)
    assert p["pair"] == pair
    assert p["head_groups"] % p["pair"] == 0


def test_forced_head_tile(lib, monkeypatch):
    monkeypatch.setenv("SMLA_HEAD_TILE", "32")
    assert smla.smla_plan_for(shape(), num_sms=152)["head_tile"] == 32
    monkeypatch.setenv("SMLA_HEAD_TILE", "64")
    assert smla.smla_plan_for(shape(heads=48), num_sms=152)["head_tile"] == 16  # 64 does not divide 48


def test_forced_splits(lib, monkeypatch):
    monkeypatch.setenv("SMLA_SPLITS", "5")
    assert smla.smla_plan_for(shape(), num_sms=152)["splits"] == 4  # 16 chunks: 4 x 4 ... no empty split
    monkeypatch.setenv("SMLA_SPLITS", "16")
    p = smla.smla_plan_for(shape(), num_sms=152)
    assert (p["splits"], p["pair"]) == (16, 1)  # one chunk per CTA: unpaired
    monkeypatch.setenv("SMLA_PAIR", "1")
    p = smla.smla_plan_for(shape(), num_sms=152)
    assert (p["splits"], p["pair"]) == (8, 2)  # forced pairing: clusters of 2 x 8 at most
    monkeypatch.delenv("SMLA_PAIR")
    monkeypatch.setenv("SMLA_SPLITS", "99")
    assert smla.smla_plan_for(shape(width=300), num_sms=152)["splits"] == 3


@pytest.mark.parametrize("kw,code", [
    (dict(heads=24), smla.EINVAL),
    (dict(heads=0), smla.EINVAL),
    (dict(head_dim=256), smla.EUNSUPPORTED),
    (dict(tokens=-1), smla.EINVAL),
    (dict(num_pools=3), smla.EUNSUPPORTED),
    (dict(num_pools=2, pool_split=4096), smla.EINVAL),
])
def test_plan_rejects_bad_shapes(lib, kw, code):
    with pytest.raises(smla.SmlaError) as e:
        smla.smla_plan_for(shape(**kw), num_sms=152)
    assert e.value.code == code


def test_decode_rejects_bad_arguments_without_launching(lib):
    s = shape(tokens=2, heads=16, width=8)
    pools = (smla.SmlaPool * 1)()
    pools[0].data, pools[0].rows, pools[0].row_bytes = 4096, 10, 576
    fake = ctypes.c_void_p(4096)
    call = lambda sh, q=fake, p=pools: lib.smla_decode(  # noqa: E731
        ctypes.byref(sh), q, p, fake, fake, None, 1.0, 1.0, 1.0, fake, None, None)
    assert call(s, q=None) == smla.EINVAL
    assert call(s, q=ctypes.c_void_p(4097)) == smla.EINVAL  # unaligned q
    bad = smla.make_shape(2, 16, 8, 576, q_strides=(16 * 576, 8))
    assert call(bad) == smla.EINVAL
    pools[0].row_bytes = 512
    assert call(s) == smla.EINVAL  # pool row bytes != head_dim
    pools[0].row_bytes = 576
    assert lib.smla_decode(ctypes.byref(smla.make_shape(0, 16, 8, 576)), None, None, None, None, None,
                           1.0, 1.0, 1.0, None, None, None) == smla.OK  # nothing to do
    assert lib.smla_error_string(smla.EINVAL).startswith(b"invalid")


def _merge_shape(**kw):
    s = smla.SmlaMergeShape()
    base = dict(sources=2, tokens=3, heads=16, reserved=0, part_stride_source=3 * 16 * 512,
                part_stride_token=16 * 512, part_stride_head=512, lse_stride_source=48, lse_stride_token=16,
                out_stride_token=16 * 512, out_stride_head=512, lse_out_stride_token=16)
    base.update(kw)
    for k, v in base.items():
        setattr(s, k, v)
    return s


@pytest.mark.parametrize("kw,ptrs", [
    (dict(sources=-1), (16, 16, 16)),
    (dict(part_stride_head=500), (16, 16, 16)),       # rows not 16-byte aligned
    (dict(out_stride_token=12), (16, 16, 16)),
    (dict(out_stride_head=256), (16, 16, 16)),        # heads overlap
    (dict(), (0, 16, 16)),                            # no parts
    (dict(), (16, 16, 0)),                            # no out
    (dict(), (8, 16, 16)),                            # parts misaligned
])
def test_merge_rejects_bad_arguments_before_any_launch(lib, kw, ptrs):
    parts, lses, out = (ctypes.c_void_p(p) if p else None for p in ptrs)
    rc = lib.smla_merge(ctypes.byref(_merge_shape(**kw)), parts, lses, None, out, None, None)
    assert rc == smla.EINVAL


def test_merge_of_nothing_is_ok_without_a_device(lib):
    assert lib.smla_merge(ctypes.byref(_merge_shape(tokens=0)), None, None, None, None, None, None) == smla.OK


def _value_shape(**kw):
    s = smla.SmlaValueShape()
    base = dict(tokens=3, heads=4, latent_stride_token=4 * 512, latent_stride_head=512,
                gate_stride_token=4 * 128, out_stride_token=4 * 128)
    base.update(kw)
    for k, v in base.items():
        setattr(s, k, v)
    return s


@pytest.mark.parametrize("kw,ptrs", [
    (dict(tokens=-1), (16, 16, 16, 16)),
    (dict(latent_stride_head=0), (16, 16, 16, 16)),
    (dict(latent_stride_token=100), (16, 16, 16, 16)),  # rows not 16-byte aligned
    (dict(gate_stride_token=4 * 128 - 8), (16, 16, 16, 16)),
    (dict(out_stride_token=4 * 128 - 8), (16, 16, 16, 16)),  # output rows overlap
    (dict(), (0, 16, 16, 16)),                           # no latent
    (dict(), (16, 16, 16, 0)),                           # no out
    (dict(), (16, 8, 16, 16)),                           # w_uv misaligned
    (dict(), (16, 16, 24, 16)),                          # gate misaligned
])
def test_value_gate_rejects_bad_arguments_before_any_launch(lib, kw, ptrs):
    latent, w, gate, out = (ctypes.c_void_p(p) if p else None for p in ptrs)
    rc = lib.smla_value_gate(ctypes.byref(_value_shape(**kw)), latent, w, gate, None, out, None)
    assert rc == smla.EINVAL


def test_value_gate_of_nothing_is_ok_without_a_device(lib):
    assert lib.smla_value_gate(ctypes.byref(_value_shape(tokens=0)), None, None, None, None, None, None) == smla.OK
    assert lib.smla_value_gate(ctypes.byref(_value_shape(heads=0)), None, None, None, None, None, None) == smla.OK


def _merge_value_shape(**kw):
    s = smla.SmlaMergeValueShape()
    base = dict(sources=2, tokens=3, heads=4, part_stride_source=3 * 4 * 512, part_stride_token=4 * 512,
                part_stride_head=512, lse_stride_source=12, lse_stride_token=4, gate_stride_token=4 * 128,
                out_stride_token=4 * 128)
    base.update(kw)
    for k, v in base.items():
        setattr(s, k, v)
    return s


@pytest.mark.parametrize("kw,ptrs", [
    (dict(sources=-1), (16, 16, 16, 16, 16)),
    (dict(part_stride_head=500), (16, 16, 16, 16, 16)),   # rows not 16-byte aligned
    (dict(lse_stride_token=-4), (16, 16, 16, 16, 16)),
    (dict(out_stride_token=4 * 128 - 8), (16, 16, 16, 16, 16)),
    (dict(), (0, 16, 16, 16, 16)),                         # no parts
    (dict(), (16, 0, 16, 16, 16)),                         # no lses
    (dict(), (8, 16, 16, 16, 16)),                         # parts misaligned
    (dict(), (16, 16, 16, 16, 0)),                         # no out
    (dict(), (16, 16, 8, 16, 16)),                         # w_uv misaligned
])
def test_merge_value_rejects_bad_arguments_before_any_launch(lib, kw, ptrs):
    parts, lses, w, gate, out = (ctypes.c_void_p(p) if p else None for p in ptrs)
    rc = lib.smla_merge_value(ctypes.byref(_merge_value_shape(**kw)), parts, lses, None, w, gate, out, None)
    assert rc == smla.EINVAL


def test_merge_value_of_nothing_is_ok_without_a_device(lib):
    assert lib.smla_merge_value(ctypes.byref(_merge_value_shape(tokens=0)), None, None, None, None, None, None,
                                None) == smla.OK


def test_merge_value_beyond_64_sources_is_unsupported_before_any_launch(lib):
    # every other argument valid: the parts of 65 sources x 3 tokens x 4 heads
    # x 512 latents, 16-byte aligned pointers, so the source limit alone refuses
    s = _merge_value_shape(sources=65, part_stride_source=3 * 4 * 512, part_stride_token=4 * 512,
                           part_stride_head=512)
    p16 = ctypes.c_void_p(16)
    rc = lib.smla_merge_value(ctypes.byref(s), p16, p16, None, p16, p16, p16, None)
    assert rc == smla.EUNSUPPORTED
    # with no tokens there is nothing to launch, whatever the source count
    s.tokens = 0
    assert lib.smla_merge_value(ctypes.byref(s), p16, p16, None, p16, p16, p16, None) == smla.OK


def test_read_device_error_needs_somewhere_to_put_the_bits(lib):
    assert lib.smla_read_device_error(None, None) == smla.EINVAL
    assert lib.smla_device_error(None) == smla.EINVAL


@pytest.mark.parametrize("limit", [0, 999, 1000000001, -5])
def test_bounded_wait_selftest_rejects_limits_outside_a_microsecond_to_a_second(lib, limit):
    assert lib.smla_selftest_bounded_wait(0, limit, None) == smla.EINVAL


def test_peak_library_exports_its_benchmarks_and_rejects_bad_arguments_without_a_device():
    path = build.build() and build.PEAK_LIBRARY
    peak = ctypes.CDLL(path)
    peak.smla_peak_mma.argtypes = [ctypes.c_int] * 6 + [ctypes.c_void_p, ctypes.c_void_p]
    peak.smla_peak_gather.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_longlong,
                                      ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    out = ctypes.c_float(0.0)
    cycles = ctypes.c_longlong(0)
    assert peak.smla_peak_mma(1, 64, 0, 0, 0, 1, ctypes.byref(cycles), ctypes.byref(out)) == -1  # no iterations
    assert peak.smla_peak_mma(2, 128, 0, 0, 10, 3, ctypes.byref(cycles), ctypes.byref(out)) == -1  # odd pair count
    peak.smla_peak_mma_chains.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_void_p]
    assert peak.smla_peak_mma_chains(1, 64, 0, 0, 3, 10, 1, ctypes.byref(cycles), ctypes.byref(out)) == -1  # 3 chains
    assert peak.smla_peak_mma_chains(2, 128, 0, 0, 2, 10, 2, ctypes.byref(cycles), ctypes.byref(out)) == -1  # pair
    assert peak.smla_peak_mma_chains(1, 64, 0, 0, 2, 0, 1, ctypes.byref(cycles), ctypes.byref(out)) == -1  # no work
    p16 = ctypes.c_void_p(16)
    assert peak.smla_peak_gather(0, 7, None, 100, p16, 2, 1, p16, ctypes.byref(out)) == -2  # no pool
    assert peak.smla_peak_gather(2, 7, p16, 100, p16, 3, 1, p16, ctypes.byref(out)) == -2  # pairs need even CTAs
    assert peak.smla_peak_gather(0, 7, ctypes.c_void_p(24), 100, p16, 2, 1, p16, ctypes.byref(out)) == -2  # unaligned


def _ds_shape(**kw):
    s = smla.SmlaDsMlaShape()
    base = dict(tokens=2, heads=64, width=100, num_pools=1, pool_split=0, q_stride_token=64 * 512, q_stride_head=512,
                rope_stride_token=64 * 64, rope_stride_head=64, idx_stride_token=100, out_stride_token=64 * 512,
                out_stride_head=512, lse_stride_token=64)
    base.update(kw)
    for k, v in base.items():
        setattr(s, k, v)
    return s


@pytest.mark.parametrize("kw,row_bytes,ptr", [
    (dict(heads=48), 656, 16),               # heads not a multiple of 32
    (dict(q_stride_head=520), 656, 16),      # q rows not 16-byte aligned
    (dict(rope_stride_head=60), 656, 16),    # rope rows below 64 values
    (dict(idx_stride_token=99), 656, 16),    # index rows shorter than the width
    (dict(num_pools=2, pool_split=101), 656, 16),
    (dict(), 576, 16),                       # a 576-byte pool
    (dict(), 656, 8),                        # misaligned q
    (dict(head_tile=48), 656, 16),           # heads per CTA neither 32 nor 64
    (dict(heads=96, head_tile=64), 656, 16),  # 64-head tiles of 96 heads
])
def test_ds_mla_decode_rejects_bad_arguments_before_any_launch(lib, kw, row_bytes, ptr):
    pools = (smla.SmlaPool * 2)()
    for i in range(2):
        pools[i].data, pools[i].rows, pools[i].row_bytes = 16, 10, row_bytes
    p = ctypes.c_void_p(ptr)
    p16 = ctypes.c_void_p(16)
    rc = lib.smla_decode_ds_mla(ctypes.byref(_ds_shape(**kw)), p, p16, pools, p16, p16, None, 0.1, 1.0, p16, None,
                                None)
    assert rc == smla.EINVAL


def test_ds_mla_decode_limits_and_empty_calls(lib):
    pools = (smla.SmlaPool * 1)()
    pools[0].data, pools[0].rows, pools[0].row_bytes = 16, 10, 656
    p16 = ctypes.c_void_p(16)
    args = (p16, p16, pools, p16, p16, None, 0.1, 1.0, p16, None, None)
    assert lib.smla_decode_ds_mla(ctypes.byref(_ds_shape(heads=1056)), *args) == smla.EUNSUPPORTED
    assert lib.smla_decode_ds_mla(ctypes.byref(_ds_shape(num_pools=3)), *args) == smla.EUNSUPPORTED
    assert lib.smla_decode_ds_mla(ctypes.byref(_ds_shape(tokens=0)), *args) == smla.OK  # nothing to launch
    bad_scale = (p16, p16, pools, p16, p16, None, -0.1, 1.0, p16, None, None)
    assert lib.smla_decode_ds_mla(ctypes.byref(_ds_shape()), *bad_scale) == smla.EINVAL


def test_ds_mla_head_tile_rule_without_a_device(lib):
    """64 heads per CTA where H allows it and the grid takes fewer waves of the
    SMs than with 32; a forced tile wins; shapes the decode rejects are
    rejected the same way."""
    def tile(**kw):
        return lib.smla_ds_mla_head_tile(ctypes.byref(_ds_shape(**kw)), 152)
    assert tile(tokens=64, heads=128) == 64      # 256 CTAs of 32 heads: 2 waves; 128 of 64: 1
    assert tile(tokens=1, heads=128) == 32       # 4 or 2 CTAs: one wave either way
    assert tile(tokens=76, heads=128) == 64      # 304 CTAs of 32: 2 waves; 152 of 64: 1
    assert tile(tokens=38, heads=128) == 32      # 152 CTAs of 32: already one wave
    assert tile(tokens=256, heads=128) == 64     # 7 waves against 4
    assert tile(tokens=64, heads=96) == 32       # 96 heads do not split into 64-head tiles
    assert tile(tokens=64, heads=128, head_tile=32) == 32
    assert tile(tokens=1, heads=64, head_tile=64) == 64
    assert tile(tokens=1, heads=96, head_tile=64) == smla.EINVAL
    assert tile(tokens=1, heads=64, head_tile=16) == smla.EINVAL
    assert tile(tokens=1, heads=48) == smla.EINVAL
    assert smla.smla_ds_mla_head_tile(64, 128, num_sms=152) == 64


def test_every_plan_over_a_grid_fits_the_hardware_and_covers_the_keys(lib):
    """Invariants of the planner over a grid of shapes (no device: 152 SMs):
    a head tile that divides H, a chunk of 96 keys only on 32/64-head tiles,
    every key covered by exactly the splits that have work, a cluster of at
    most 16 CTAs, pairing only of an even number of head groups over one pool,
    and one CTA's shared memory and TMEM within the SM's."""
    seen_chunks, seen_pairs = set(), set()
    for tokens in (1, 2, 5, 12, 33, 64, 128, 300):
        for heads in (16, 32, 48, 64, 96, 128, 256):
            for width in (1, 95, 96, 128, 129, 640, 1000, 2048, 4096):
                for dim, pools in ((576, 1), (512, 1), (576, 2)):
                    split_col = min(width, 128) if pools == 2 else 0
                    p = smla.smla_plan_for(smla.make_shape(tokens, heads, width, dim, pools, split_col), num_sms=152)
                    where = (tokens, heads, width, dim, pools, p)
                    tile = p["head_tile"]
                    assert tile in (16, 32, 64) and heads % tile == 0 and p["head_groups"] * tile == heads, where
                    assert p["chunk"] in (96, 128) and (p["chunk"] == 128 or tile >= 32), where
                    assert p["chunks"] == -(-width // p["chunk"]), where
                    assert 1 <= p["splits"] <= 16, where
                    assert p["splits"] * p["chunks_per_split"] >= p["chunks"], where
                    assert (p["splits"] - 1) * p["chunks_per_split"] < max(p["chunks"], 1), where
                    assert p["pair"] in (1, 2) and p["pair"] * p["splits"] <= 16, where
                    if p["pair"] == 2:
                        assert p["head_groups"] % 2 == 0 and pools == 1, where
                    assert p["ctas"] == tokens * p["head_groups"] * p["splits"], where
                    assert p["threads"] == 512 and p["smem_bytes"] <= 227 * 1024, where
                    cols = p["tmem_columns"]
                    assert 32 <= cols <= 512 and cols & (cols - 1) == 0, where
                    seen_chunks.add(p["chunk"])
                    seen_pairs.add(p["pair"])
    assert seen_chunks == {96, 128} and seen_pairs == {1, 2}  # the grid reaches every kind of plan
