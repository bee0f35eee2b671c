"""Seeded synthetic inputs for sparse MLA decode.

This module only draws inputs: it holds none of the decode arithmetic, and both
the CPU oracle (in tests) and the CUDA path take their inputs from it.

Shapes and distributions follow the workloads the pages describe (DeepSeek-V4.1
``sparse_mla_cute`` module docstring, "The problem": 16 heads, 512-byte rows,
128 sliding-window columns then top-k columns of a compressed pool, -1 holes,
per-token counts; Kimi K3.1 ``attn_sparse`` module docstring, "Why": 5 verify
rows, ~256 keys per row, 576-byte rows = 512 latent + 64 rope, per-tensor FP8
scale).  Every value is drawn from numpy's PCG64 generator, which gives the same
stream on every platform; E4M3 bytes are N(0, 1) draws rounded by torch's
float8_e4m3fn cast (|x| < 448 never saturates).

A workload is a dict:
  q          uint8 [T, H, D]        E4M3 query bytes
  pools      list of uint8 [R, D]   E4M3 KV rows (1 or 2 pools)
  pool_split int                    columns below it index pool 0, others pool 1
  indices    int32 [T, W]           row per column, -1 = hole
  lens       int32 [T]              active count per token
  sinks      float32 [H] or None    per-head sink, in score units
  bmm1_scale, bmm2_scale, k_scale   floats
  name       str
"""

from __future__ import annotations

import math

import numpy as np
import torch

LATENT = 512


def e4m3_normal(rng: np.random.Generator, shape, block: int = 1 << 24) -> np.ndarray:
    """E4M3 bytes of N(0, 1) draws, generated in blocks to bound host memory."""
    total = int(np.prod(shape))
    out = np.empty(total, np.uint8)
    for start in range(0, total, block):
        n = min(block, total - start)
        x = rng.standard_normal(n, dtype=np.float32)
        out[start:start + n] = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return out.reshape(shape)


def unique_rows(rng: np.random.Generator, pool_rows: int, k: int,
                exclude: np.ndarray | None = None) -> np.ndarray:
    """k distinct row ids in [0, pool_rows), uniform, avoiding ``exclude``."""
    if k == 0:
        return np.zeros(0, np.int64)
    if pool_rows <= 4 * k + (0 if exclude is None else exclude.size):
        candidates = np.arange(pool_rows)
        if exclude is not None:
            candidates = np.setdiff1d(candidates, exclude, assume_unique=False)
        return rng.choice(candidates, size=k, replace=False)
    chosen = np.zeros(0, np.int64)
    banned = set() if exclude is None else set(exclude.tolist())
    while chosen.size < k:
        draw = rng.integers(0, pool_rows, size=2 * (k - chosen.size))
        draw = np.array([d for d in draw if d not in banned], np.int64)
        chosen = np.unique(np.concatenate([chosen, draw]))
    keep = rng.permutation(chosen.size)[:k]
    return rng.permutation(chosen[keep])


def _base(name, rng, T, H, D, pool_rows_list, W):
    return {
        "name": name,
        "q": e4m3_normal(rng, (T, H, D)),
        "pools": [e4m3_normal(rng, (r, D)) for r in pool_rows_list],
        "pool_split": 0,
        "indices": np.full((T, W), -1, np.int32),
        "lens": np.zeros(T, np.int32),
        "sinks": None,
        "bmm1_scale": 1.0 / math.sqrt(192.0),
        "bmm2_scale": 1.0,
        "k_scale": 1.0,
    }


def tiny(seed: int = 1000) -> dict:
    """1 token x 16 heads x 576-byte rows; 4096-row pool; 256 unique indices,
    all active; softmax scale 1/sqrt(192); no sinks."""
    rng = np.random.default_rng(seed)
    w = _base("tiny_t1_h16_k256_d576", rng, 1, 16, 576, [4096], 256)
    w["indices"][0] = unique_rows(rng, 4096, 256)
    w["lens"][:] = 256
    return w


def verify_rows(seed: int = 1001) -> dict:
    """5 verify rows x 128 heads x 576-byte rows; 65536-row pool, k_scale 0.05;
    counts drawn from {0} U {64..256}, one row forced to 0; unique indices
    padded with -1 to width 256."""
    rng = np.random.default_rng(seed)
    T, W = 5, 256
    w = _base("verify_t5_h128_k256_d576", rng, T, 128, 576, [65536], W)
    w["k_scale"] = 0.05
    w["bmm1_scale"] = 0.05 / math.sqrt(192.0)
    choices = np.concatenate([[0], np.arange(64, 257)])
    counts = rng.choice(choices, size=T)
    counts[2] = 0
    for t in range(T):
        w["indices"][t, : counts[t]] = unique_rows(rng, 65536, int(counts[t]))
    w["lens"][:] = counts
    return w


def two_pool_sinks(seed: int = 1002) -> dict:
    """12 tokens x 16 heads x 512-byte rows; width 640: columns 0..127 index an
    8192-row sliding-window pool, 128..639 a 262144-row compressed pool; 5% of
    the indices set to -1; lens uniform in 300..640; sinks N(0, 1);
    bmm1_scale = 1/sqrt(512), bmm2_scale = 0.5."""
    rng = np.random.default_rng(seed)
    T, W, split = 12, 640, 128
    w = _base("two_pool_t12_h16_w640_d512", rng, T, 16, 512, [8192, 262144], W)
    w["pool_split"] = split
    w["bmm1_scale"] = 1.0 / math.sqrt(512.0)
    w["bmm2_scale"] = 0.5
    for t in range(T):
        w["indices"][t, :split] = rng.integers(0, 8192, size=split)
        w["indices"][t, split:] = rng.integers(0, 262144, size=W - split)
    holes = rng.random((T, W)) < 0.05
    w["indices"][holes] = -1
    w["lens"][:] = rng.integers(300, 641, size=T)
    w["sinks"] = rng.standard_normal(16, dtype=np.float32)
    return w


def bandwidth_batch(seed: int = 1003, tokens: int = 64, heads: int = 128, topk: int = 2048,
                    pool_rows: int = 1 << 20, hot_rows: int = 20000, pool=None) -> dict:
    """64 tokens x 128 heads x 2048 keys on a 1,048,576 x 576-byte pool. Per
    token half of the rows come from a common 20k-row hot set (so ~50% of the
    rows are shared across tokens), half from the rest; all active; no sinks.
    ``pool`` reuses an already drawn pool (the rotation sets of a benchmark)."""
    rng = np.random.default_rng(seed)
    D, W = 576, topk
    w = {
        "name": f"batch_t{tokens}_h{heads}_k{topk}_d576",
        "q": e4m3_normal(rng, (tokens, heads, D)),
        "pools": [e4m3_normal(rng, (pool_rows, D)) if pool is None else pool],
        "pool_split": 0,
        "indices": np.full((tokens, W), -1, np.int32),
        "lens": np.full(tokens, W, np.int32),
        "sinks": None,
        "bmm1_scale": 1.0 / math.sqrt(192.0),
        "bmm2_scale": 1.0,
        "k_scale": 1.0,
    }
    hot = unique_rows(rng, pool_rows, hot_rows)
    for t in range(tokens):
        a = rng.choice(hot, size=W // 2, replace=False)
        b = unique_rows(rng, pool_rows, W - W // 2, exclude=hot)
        w["indices"][t] = rng.permutation(np.concatenate([a, b]))
    return w


def sweep_point(tokens: int, heads: int, topk: int, seed: int | None = None,
                pool=None, pool_rows: int = 1 << 20) -> dict:
    """One point of the sweep: 576-byte rows N(0, 1) in a 1M-row pool, unique
    uniform indices, 10% -1 holes, counts uniform in [k/2, k]."""
    if seed is None:
        seed = 2000 + 7919 * tokens + 104729 * heads + topk
    rng = np.random.default_rng(seed)
    D, W = 576, topk
    w = {
        "name": f"sweep_t{tokens}_h{heads}_k{topk}_d576",
        "q": e4m3_normal(rng, (tokens, heads, D)),
        "pools": [e4m3_normal(rng, (pool_rows, D)) if pool is None else pool],
        "pool_split": 0,
        "indices": np.full((tokens, W), -1, np.int32),
        "lens": rng.integers(topk // 2, topk + 1, size=tokens).astype(np.int32),
        "sinks": None,
        "bmm1_scale": 1.0 / math.sqrt(192.0),
        "bmm2_scale": 1.0,
        "k_scale": 1.0,
    }
    rows = w["pools"][0].shape[0]
    for t in range(tokens):
        w["indices"][t] = unique_rows(rng, rows, W)
    holes = rng.random((tokens, W)) < 0.10
    w["indices"][holes] = -1
    return w


SWEEP_TOKENS = (1, 2, 6, 12, 32, 128, 256)
SWEEP_HEADS = (16, 64, 128)
SWEEP_TOPK = (256, 512, 1024, 2048)

CONFIGS = {
    "tiny": tiny,
    "verify": verify_rows,
    "two_pool": two_pool_sinks,
    "batch": bandwidth_batch,
}


def small(name: str, seed: int, tokens: int, heads: int, width: int, head_dim: int,
          pool_rows: int = 512, holes: float = 0.0, lens=None, sinks: bool = False,
          two_pools: bool = False, pool_split: int = 0, k_scale: float = 1.0,
          bmm2_scale: float = 1.0, duplicates: bool = False) -> dict:
    """A small random problem for parity and edge-case tests."""
    rng = np.random.default_rng(seed)
    w = {
        "name": name,
        "q": e4m3_normal(rng, (tokens, heads, head_dim)),
        "pools": [e4m3_normal(rng, (pool_rows, head_dim))],
        "pool_split": 0,
        "sinks": rng.standard_normal(heads, dtype=np.float32) if sinks else None,
        "bmm1_scale": 1.0 / math.sqrt(192.0 if head_dim == 576 else 512.0),
        "bmm2_scale": bmm2_scale,
        "k_scale": k_scale,
    }
    if two_pools:
        w["pools"].append(e4m3_normal(rng, (pool_rows * 2, head_dim)))
        w["pool_split"] = pool_split
    idx = np.empty((tokens, width), np.int32)
    for t in range(tokens):
        if duplicates:
            idx[t] = rng.integers(0, pool_rows, size=width)
        elif two_pools:
            idx[t, :pool_split] = rng.integers(0, pool_rows, size=min(pool_split, width))
            idx[t, pool_split:] = rng.integers(0, 2 * pool_rows, size=max(0, width - pool_split))
        else:
            idx[t] = unique_rows(rng, pool_rows, width) if width <= pool_rows else \
                rng.integers(0, pool_rows, size=width)
    if holes > 0:
        idx[rng.random((tokens, width)) < holes] = -1
    w["indices"] = idx
    if lens is None:
        w["lens"] = np.full(tokens, width, np.int32)
    else:
        w["lens"] = np.asarray(lens, np.int32).reshape(tokens)
    return w


def unique_active_rows(w: dict) -> int:
    """Distinct (pool, row) pairs that the active columns of ``w`` touch."""
    T, W = w["indices"].shape
    seen = []
    for pool_id in range(len(w["pools"])):
        rows = []
        for t in range(T):
            n = max(0, min(int(w["lens"][t]), W))
            cols = np.arange(n)
            if len(w["pools"]) == 2:
                cols = cols[cols >= w["pool_split"]] if pool_id == 1 else cols[cols < w["pool_split"]]
            r = w["indices"][t, cols]
            r = r[(r >= 0) & (r < w["pools"][pool_id].shape[0])]
            rows.append(r)
        seen.append(np.unique(np.concatenate(rows)).size if rows else 0)
    return int(sum(seen))


def merge_sets(seed: int = 1005, sources: int = 8, tokens: int = 64, heads: int = 128, device=None):
    """Partial (out, lse) sets of one decode step split over ``sources`` key
    shards (a DCP8 step of the 64 x 128 batch by default): BF16 rows N(0, 1),
    base-2 LSEs U(4, 12), 3 % of the (source, token, head) entries empty
    (LSE -inf), token 5 with count 0. Torch tensors on ``device`` (a seeded
    torch generator there): parts bfloat16 [S, T, H, 512], lses float32
    [S, T, H], lens int32 [T]."""
    import torch

    device = torch.device(device or "cpu")
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    parts = torch.randn((sources, tokens, heads, 512), generator=gen, device=device).to(torch.bfloat16)
    lses = torch.rand((sources, tokens, heads), generator=gen, device=device) * 8.0 + 4.0
    empty = torch.rand((sources, tokens, heads), generator=gen, device=device) < 0.03
    lses = torch.where(empty, torch.full_like(lses, float("-inf")), lses)
    lens = torch.full((tokens,), 2048, dtype=torch.int32, device=device)
    if tokens > 5:
        lens[5] = 0
    return parts, lses, lens


# ------------------------------------------------------------ fp8_ds_mla rows
# A 656-byte cache row (Kimi K3.1 dsa_indexer_mxfp4 page: mla_cache of
# [num_blocks, block_size, 656] bytes, viewed as FP8, float32 and BF16), laid
# out as this library reads it: 512 E4M3 latent codes, four little-endian FP32
# scales, 64 little-endian BF16 rope values.
DS_MLA_ROW = 656


def bf16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    """uint16 BF16 bits of N(0, 1) draws (torch's round-to-nearest cast)."""
    x = rng.standard_normal(int(np.prod(shape)), dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(shape)


def ds_mla_rows(rng: np.random.Generator, rows: int, block: int = 1 << 16) -> np.ndarray:
    """uint8 [rows, 656]: N(0, 1) E4M3 codes, four scales 2^u * v (u uniform in
    [-6, 2], v uniform in [0.5, 1)), N(0, 1) BF16 rope values."""
    out = np.empty((rows, DS_MLA_ROW), np.uint8)
    for start in range(0, rows, block):
        n = min(block, rows - start)
        out[start:start + n, :512] = e4m3_normal(rng, (n, 512))
        scales = (2.0 ** rng.integers(-6, 3, (n, 4)) * rng.uniform(0.5, 1.0, (n, 4))).astype("<f4")
        out[start:start + n, 512:528] = scales.view(np.uint8).reshape(n, 16)
        out[start:start + n, 528:] = bf16_normal(rng, (n, 64)).astype("<u2").view(np.uint8).reshape(n, 128)
    return out


def ds_mla_small(name: str, seed: int, tokens: int, heads: int, width: int, pool_rows: int = 512,
                 holes: float = 0.0, lens=None, sinks: bool = False, two_pools: bool = False,
                 pool_split: int = 0, bmm2_scale: float = 1.0) -> dict:
    """A small random problem over fp8_ds_mla rows. Keys of the dict as for the
    576-byte workloads, except: q_latent uint8 [T, H, 512] E4M3 bytes and
    q_rope uint16 [T, H, 64] BF16 bits instead of q; pools of [R, 656] rows; no
    k_scale."""
    rng = np.random.default_rng(seed)
    w = {
        "name": name,
        "q_latent": e4m3_normal(rng, (tokens, heads, 512)),
        "q_rope": bf16_normal(rng, (tokens, heads, 64)),
        "pools": [ds_mla_rows(rng, pool_rows)],
        "pool_split": 0,
        "sinks": rng.standard_normal(heads, dtype=np.float32) if sinks else None,
        "bmm1_scale": 1.0 / math.sqrt(192.0),
        "bmm2_scale": bmm2_scale,
    }
    if two_pools:
        w["pools"].append(ds_mla_rows(rng, pool_rows * 2))
        w["pool_split"] = pool_split
    idx = np.empty((tokens, width), np.int32)
    for t in range(tokens):
        if two_pools:
            idx[t, :pool_split] = rng.integers(0, pool_rows, size=min(pool_split, width))
            idx[t, pool_split:] = rng.integers(0, 2 * pool_rows, size=max(0, width - pool_split))
        else:
            idx[t] = unique_rows(rng, pool_rows, width) if width <= pool_rows else \
                rng.integers(0, pool_rows, size=width)
    if holes > 0:
        idx[rng.random((tokens, width)) < holes] = -1
    w["indices"] = idx
    w["lens"] = np.full(tokens, width, np.int32) if lens is None else np.asarray(lens, np.int32).reshape(tokens)
    return w


def ds_mla_batch(seed: int = 1007, tokens: int = 64, heads: int = 128, topk: int = 2048, pool_rows: int = 1 << 20,
                 hot_rows: int = 20000, pool=None) -> dict:
    """The 64 x 128 x 2048 bandwidth batch over fp8_ds_mla rows: the same
    index recipe as ``bandwidth_batch`` (half of each token's rows from a
    common 20k-row hot set), a 1,048,576 x 656-byte pool, no sinks."""
    rng = np.random.default_rng(seed)
    W = topk
    w = {
        "name": f"ds_mla_batch_t{tokens}_h{heads}_k{topk}_r656",
        "q_latent": e4m3_normal(rng, (tokens, heads, 512)),
        "q_rope": bf16_normal(rng, (tokens, heads, 64)),
        "pools": [ds_mla_rows(rng, pool_rows) if pool is None else pool],
        "pool_split": 0,
        "indices": np.full((tokens, W), -1, np.int32),
        "lens": np.full(tokens, W, np.int32),
        "sinks": None,
        "bmm1_scale": 1.0 / math.sqrt(192.0),
        "bmm2_scale": 1.0,
    }
    hot = unique_rows(rng, pool_rows, hot_rows)
    for t in range(tokens):
        a = rng.choice(hot, size=W // 2, replace=False)
        b = unique_rows(rng, pool_rows, W - W // 2, exclude=hot)
        w["indices"][t] = rng.permutation(np.concatenate([a, b]))
    return w
