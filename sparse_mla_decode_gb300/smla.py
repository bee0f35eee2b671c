"""Python binding of libsmla.so: argument marshalling only.

The names mirror the C ABI in ``include/smla.h``. Every step of the decode runs
in the library's CUDA kernels; when the library is missing this module raises
instead of computing anything itself.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

OK, EINVAL, EUNSUPPORTED, ECUDA, EDEVICE = 0, -1, -2, -3, -4
DEV_INDEX_RANGE, DEV_TIMEOUT = 1, 2
LATENT = 512

_lock = threading.Lock()
_lib = None


class SmlaPool(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("row_bytes", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class SmlaDsMlaShape(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int32), ("heads", ctypes.c_int32), ("width", ctypes.c_int32),
        ("num_pools", ctypes.c_int32), ("pool_split", ctypes.c_int32), ("head_tile", ctypes.c_int32),
        ("q_stride_token", ctypes.c_int64), ("q_stride_head", ctypes.c_int64),
        ("rope_stride_token", ctypes.c_int64), ("rope_stride_head", ctypes.c_int64),
        ("idx_stride_token", ctypes.c_int64),
        ("out_stride_token", ctypes.c_int64), ("out_stride_head", ctypes.c_int64),
        ("lse_stride_token", ctypes.c_int64),
    ]


class SmlaShape(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int32), ("heads", ctypes.c_int32), ("width", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("num_pools", ctypes.c_int32), ("pool_split", ctypes.c_int32),
        ("q_stride_token", ctypes.c_int64), ("q_stride_head", ctypes.c_int64),
        ("idx_stride_token", ctypes.c_int64),
        ("out_stride_token", ctypes.c_int64), ("out_stride_head", ctypes.c_int64),
        ("lse_stride_token", ctypes.c_int64),
    ]


class SmlaPlan(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "head_tile", "head_groups", "chunk", "chunks", "splits", "chunks_per_split", "ctas",
        "threads", "smem_bytes", "tmem_columns", "num_sms", "resident_ctas", "pair")]


class SmlaMergeShape(ctypes.Structure):
    _fields_ = [
        ("sources", ctypes.c_int32), ("tokens", ctypes.c_int32), ("heads", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("part_stride_source", ctypes.c_int64), ("part_stride_token", ctypes.c_int64),
        ("part_stride_head", ctypes.c_int64),
        ("lse_stride_source", ctypes.c_int64), ("lse_stride_token", ctypes.c_int64),
        ("out_stride_token", ctypes.c_int64), ("out_stride_head", ctypes.c_int64),
        ("lse_out_stride_token", ctypes.c_int64),
    ]


class SmlaMxfp4Shape(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int32), ("heads", ctypes.c_int32), ("padded_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("q_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("q_stride_token", ctypes.c_int64), ("q_stride_head", ctypes.c_int64),
        ("w_stride_token", ctypes.c_int64), ("packed_stride_token", ctypes.c_int64),
        ("scale_stride_token", ctypes.c_int64), ("w_out_stride_token", ctypes.c_int64),
    ]


class SmlaValueShape(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int32), ("heads", ctypes.c_int32), ("reserved", ctypes.c_int32 * 2),
        ("latent_stride_token", ctypes.c_int64), ("latent_stride_head", ctypes.c_int64),
        ("gate_stride_token", ctypes.c_int64), ("out_stride_token", ctypes.c_int64),
    ]


class SmlaMergeValueShape(ctypes.Structure):
    _fields_ = [
        ("sources", ctypes.c_int32), ("tokens", ctypes.c_int32), ("heads", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("part_stride_source", ctypes.c_int64), ("part_stride_token", ctypes.c_int64),
        ("part_stride_head", ctypes.c_int64),
        ("lse_stride_source", ctypes.c_int64), ("lse_stride_token", ctypes.c_int64),
        ("gate_stride_token", ctypes.c_int64), ("out_stride_token", ctypes.c_int64),
    ]


DTYPE_BF16 = 1
DTYPE_F32 = 2
VALUE_DIM = 128


class SmlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        lib = _lib
        text = lib.smla_error_string(code).decode() if lib is not None else str(code)
        if code == ECUDA and lib is not None:
            text += f" (cudaError {lib.smla_last_cuda_error()})"
        super().__init__(f"{what}: {text} [{code}]")
        self.code = code


def library_path() -> str:
    return _build.LIBRARY


def load(path: str | None = None):
    """Loads libsmla.so (built by ``sparse_mla_decode_gb300.build``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIBRARY
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m sparse_mla_decode_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(path)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        lib.smla_plan_for.argtypes = [ctypes.POINTER(SmlaShape), i32, ctypes.POINTER(SmlaPlan)]
        lib.smla_plan_for.restype = i32
        lib.smla_decode.argtypes = [ctypes.POINTER(SmlaShape), vp, ctypes.POINTER(SmlaPool), vp, vp,
                                    vp, ctypes.c_float, ctypes.c_float, ctypes.c_float, vp, vp, vp]
        lib.smla_decode.restype = i32
        lib.smla_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32)]
        lib.smla_device_error.restype = i32
        lib.smla_error_string.argtypes = [i32]
        lib.smla_error_string.restype = ctypes.c_char_p
        lib.smla_last_cuda_error.restype = i32
        lib.smla_version.restype = i32
        lib.smla_merge.argtypes = [ctypes.POINTER(SmlaMergeShape), vp, vp, vp, vp, vp, vp]
        lib.smla_merge.restype = i32
        lib.smla_mxfp4_q_quant.argtypes = [ctypes.POINTER(SmlaMxfp4Shape), vp, vp, ctypes.c_float, vp, vp, vp, vp]
        lib.smla_mxfp4_q_quant.restype = i32
        lib.smla_value_gate.argtypes = [ctypes.POINTER(SmlaValueShape), vp, vp, vp, vp, vp, vp]
        lib.smla_value_gate.restype = i32
        lib.smla_merge_value.argtypes = [ctypes.POINTER(SmlaMergeValueShape), vp, vp, vp, vp, vp, vp, vp]
        lib.smla_merge_value.restype = i32
        lib.smla_decode_ds_mla.argtypes = [ctypes.POINTER(SmlaDsMlaShape), vp, vp, ctypes.POINTER(SmlaPool), vp, vp,
                                           vp, ctypes.c_float, ctypes.c_float, vp, vp, vp]
        lib.smla_decode_ds_mla.restype = i32
        lib.smla_ds_mla_head_tile.argtypes = [ctypes.POINTER(SmlaDsMlaShape), i32]
        lib.smla_ds_mla_head_tile.restype = i32
        lib.smla_read_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        lib.smla_read_device_error.restype = i32
        lib.smla_selftest_bounded_wait.argtypes = [i32, ctypes.c_int64, vp]
        lib.smla_selftest_bounded_wait.restype = i32
        _lib = lib
        return lib


def make_shape(tokens, heads, width, head_dim, num_pools=1, pool_split=0, q_strides=None,
               idx_stride=None, out_strides=None, lse_stride=None) -> SmlaShape:
    s = SmlaShape()
    s.tokens, s.heads, s.width, s.head_dim = tokens, heads, width, head_dim
    s.num_pools, s.pool_split = num_pools, pool_split
    s.q_stride_token, s.q_stride_head = q_strides or (heads * head_dim, head_dim)
    s.idx_stride_token = width if idx_stride is None else idx_stride
    s.out_stride_token, s.out_stride_head = out_strides or (heads * LATENT, LATENT)
    s.lse_stride_token = heads if lse_stride is None else lse_stride
    return s


def smla_plan_for(shape: SmlaShape, num_sms: int = 0) -> dict:
    lib = load()
    plan = SmlaPlan()
    rc = lib.smla_plan_for(ctypes.byref(shape), int(num_sms), ctypes.byref(plan))
    if rc != OK:
        raise SmlaError(rc, "smla_plan_for")
    return {name: getattr(plan, name) for name, _ in SmlaPlan._fields_}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# Shape structs and pool descriptor arrays of recent calls, by the tuples
# that define them: a decode step repeats the same few, and building them
# anew costs more host time than the C call.
_shapes: dict = {}
_pool_arrays: dict = {}


def _cached(cache: dict, key, build):
    v = cache.get(key)
    if v is None:
        if len(cache) >= 256:
            cache.clear()
        v = cache[key] = build()
    return v


def _pool_array(kv_pools, D):
    def build():
        pools = (SmlaPool * len(kv_pools))()
        for i, pool in enumerate(kv_pools):
            if pool.shape[0] > 1 and (pool.stride(1) != 1 or pool.stride(0) != D):
                raise ValueError("pool rows must be contiguous")
            pools[i].data = pool.data_ptr()
            pools[i].rows = pool.shape[0]
            pools[i].row_bytes = pool.shape[1]
            pools[i].reserved = 0
        return pools

    key = tuple((p.data_ptr(), p.shape[0], p.shape[1], p.stride(0), p.stride(1)) for p in kv_pools)
    return _cached(_pool_arrays, (D, key), build)


def smla_decode(q: torch.Tensor, kv_pools, indices: torch.Tensor, lens: torch.Tensor,
                sinks: torch.Tensor | None, bmm1_scale: float, bmm2_scale: float, k_scale: float,
                out: torch.Tensor, lse: torch.Tensor | None, stream=None, pool_split: int = 0):
    """Sparse MLA decode through the C ABI.

    q: uint8 (E4M3 bytes) or float8_e4m3fn [T, H, D] on the device, last dim
    contiguous; kv_pools: list of 1 or 2 [rows, D] E4M3 tensors, rows
    contiguous; indices int32 [T, >= W] (W = indices.shape[1]); lens int32 [T];
    sinks float32 [H] or None; out bf16 [T, H, 512]; lse float32 [T, H] or None.
    Runs on ``stream`` (default: torch's current stream) without synchronising.
    """
    lib = _lib if _lib is not None else load()
    T, H, D = q.shape
    W = indices.shape[1]
    qst, ost, ist = q.stride(), out.stride(), indices.stride()
    if (D > 1 and qst[2] != 1) or (out.shape[2] > 1 and ost[2] != 1) or (W > 1 and ist[1] != 1):
        raise ValueError("q, out and indices: innermost dimension must be contiguous")
    esz = q.element_size()
    lse_stride = None if lse is None else lse.stride(0)
    key = (T, H, W, D, len(kv_pools), pool_split, qst[0] * esz, qst[1] * esz, ist[0], ost[0], ost[1], lse_stride)
    shape = _cached(_shapes, key, lambda: make_shape(
        T, H, W, D, len(kv_pools), pool_split, q_strides=(qst[0] * esz, qst[1] * esz), idx_stride=ist[0],
        out_strides=(ost[0], ost[1]), lse_stride=lse_stride))
    pools = _pool_array(kv_pools, D)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    rc = lib.smla_decode(shape, q.data_ptr(), pools, indices.data_ptr(), lens.data_ptr(),
                         None if sinks is None else sinks.data_ptr(), bmm1_scale, bmm2_scale, k_scale,
                         out.data_ptr(), None if lse is None else lse.data_ptr(), handle)
    if rc != OK:
        raise SmlaError(rc, "smla_decode")
    return out, lse


DS_MLA_ROW_BYTES = 656


def smla_decode_ds_mla(q_latent: torch.Tensor, q_rope: torch.Tensor, kv_pools, indices: torch.Tensor,
                       lens: torch.Tensor, sinks: torch.Tensor | None, bmm1_scale: float, bmm2_scale: float,
                       out: torch.Tensor, lse: torch.Tensor | None, stream=None, pool_split: int = 0,
                       head_tile: int = 0):
    """Sparse MLA decode over fp8_ds_mla rows through the C ABI.

    q_latent: uint8 (E4M3 bytes) or float8_e4m3fn [T, H, 512]; q_rope: bfloat16
    [T, H, 64]; kv_pools: list of 1 or 2 uint8 [rows, 656] tensors, rows
    contiguous; indices int32 [T, >= W]; lens int32 [T]; sinks float32 [H] or
    None; out bf16 [T, H, 512]; lse float32 [T, H] or None. H a multiple of 32.
    head_tile: heads per CTA, 0 (the library's choice), 32 or 64.
    """
    lib = _lib if _lib is not None else load()
    T, H, _ = q_latent.shape
    W = indices.shape[1]
    qst, rst, ost, ist = q_latent.stride(), q_rope.stride(), out.stride(), indices.stride()
    if qst[2] != 1 or rst[2] != 1 or ost[2] != 1 or (W > 1 and ist[1] != 1):
        raise ValueError("q_latent, q_rope, out and indices: innermost dimension must be contiguous")
    esz = q_latent.element_size()
    lse_stride = None if lse is None else lse.stride(0)
    key = ("ds", T, H, W, len(kv_pools), pool_split, qst[0] * esz, qst[1] * esz, rst[0], rst[1], ist[0], ost[0],
           ost[1], lse_stride, head_tile)

    def build():
        sh = SmlaDsMlaShape()
        sh.tokens, sh.heads, sh.width, sh.num_pools, sh.pool_split = T, H, W, len(kv_pools), pool_split
        sh.head_tile = head_tile
        sh.q_stride_token, sh.q_stride_head = qst[0] * esz, qst[1] * esz
        sh.rope_stride_token, sh.rope_stride_head = rst[0], rst[1]
        sh.idx_stride_token = ist[0]
        sh.out_stride_token, sh.out_stride_head = ost[0], ost[1]
        sh.lse_stride_token = lse_stride if lse_stride is not None else H
        return sh

    shape = _cached(_shapes, key, build)
    pools = _pool_array(kv_pools, DS_MLA_ROW_BYTES)
    if stream is None:
        stream = torch.cuda.current_stream(q_latent.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    rc = lib.smla_decode_ds_mla(shape, q_latent.data_ptr(), q_rope.data_ptr(), pools, indices.data_ptr(),
                                lens.data_ptr(), None if sinks is None else sinks.data_ptr(), bmm1_scale,
                                bmm2_scale, out.data_ptr(), None if lse is None else lse.data_ptr(), handle)
    if rc != OK:
        raise SmlaError(rc, "smla_decode_ds_mla")
    return out, lse


def decode_ds_mla(q_latent, q_rope, kv_pools, indices, lens, sinks=None, bmm1_scale=1.0, bmm2_scale=1.0,
                  pool_split=0, stream=None, with_lse=True, head_tile=0):
    """Allocates out (and lse) on q_latent's device and calls :func:`smla_decode_ds_mla`."""
    T, H, _ = q_latent.shape
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q_latent.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=q_latent.device) if with_lse else None
    return smla_decode_ds_mla(q_latent, q_rope, kv_pools, indices, lens, sinks, bmm1_scale, bmm2_scale, out, lse,
                              stream=stream, pool_split=pool_split, head_tile=head_tile)


def smla_ds_mla_head_tile(tokens: int, heads: int, head_tile: int = 0, num_sms: int = 0) -> int:
    """Heads per CTA that :func:`smla_decode_ds_mla` takes (C ABI; ``num_sms``
    0 asks the current device)."""
    sh = SmlaDsMlaShape()
    sh.tokens, sh.heads, sh.head_tile, sh.num_pools = tokens, heads, head_tile, 1
    rc = load().smla_ds_mla_head_tile(ctypes.byref(sh), int(num_sms))
    if rc < 0:
        raise SmlaError(rc, "smla_ds_mla_head_tile")
    return int(rc)


def smla_device_error() -> int:
    """Reads and clears the device error word (synchronises the device)."""
    lib = load()
    bits = ctypes.c_int32(0)
    rc = lib.smla_device_error(ctypes.byref(bits))
    if rc != OK:
        raise SmlaError(rc, "smla_device_error")
    return int(bits.value)


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def smla_read_device_error(stream=None) -> int:
    """Reads and clears the device error word in ``stream``'s order (the
    current stream by default) and waits for that stream alone."""
    lib = load()
    bits = ctypes.c_int32(0)
    rc = lib.smla_read_device_error(ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(bits))
    if rc != OK:
        raise SmlaError(rc, "smla_read_device_error")
    return int(bits.value)


def smla_selftest_bounded_wait(arrive: bool, limit_ns: int, stream=None) -> None:
    """Launches the bounded-wait self-test (one warp waits on an mbarrier that
    only it may arrive on) on ``stream``."""
    rc = load().smla_selftest_bounded_wait(int(bool(arrive)), int(limit_ns),
                                           ctypes.c_void_p(_stream_handle(stream)))
    if rc != OK:
        raise SmlaError(rc, "smla_selftest_bounded_wait")


def smla_version() -> int:
    return int(load().smla_version())


def decode(q, kv_pools, indices, lens, sinks=None, bmm1_scale=1.0, bmm2_scale=1.0, k_scale=1.0,
           pool_split=0, stream=None, with_lse=True):
    """Allocates the outputs on q's device and calls :func:`smla_decode`."""
    T, H, _ = q.shape
    out = torch.empty((T, H, LATENT), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=q.device) if with_lse else None
    return smla_decode(q, kv_pools, indices, lens, sinks, bmm1_scale, bmm2_scale, k_scale, out, lse,
                       stream=stream, pool_split=pool_split)


def smla_merge(parts: torch.Tensor, lses: torch.Tensor, lens: torch.Tensor | None, out: torch.Tensor,
               lse_out: torch.Tensor | None, stream=None):
    """LSE merge of partial sets through the C ABI (see ``smla_merge`` in smla.h).

    parts: bfloat16 [S, T, H, 512] on the device, latents contiguous; lses:
    float32 [S, T, H] (base 2), heads contiguous; lens: int32 [T] or None;
    out: bfloat16 [T, H, 512]; lse_out: float32 [T, H] or None. Runs on
    ``stream`` (default: torch's current stream) without synchronising."""
    lib = load()
    S, T, H, J = parts.shape
    if J != LATENT or tuple(lses.shape) != (S, T, H) or tuple(out.shape) != (T, H, LATENT):
        raise ValueError("merge: parts [S, T, H, 512], lses [S, T, H], out [T, H, 512]")
    if parts.stride(3) != 1 or out.stride(2) != 1 or (H > 1 and lses.stride(2) != 1):
        raise ValueError("merge: latents and heads must be contiguous")
    if lse_out is not None and H > 1 and lse_out.stride(1) != 1:
        raise ValueError("merge: lse_out heads must be contiguous")
    shape = SmlaMergeShape()
    shape.sources, shape.tokens, shape.heads, shape.reserved = S, T, H, 0
    shape.part_stride_source, shape.part_stride_token, shape.part_stride_head = parts.stride()[:3]
    shape.lse_stride_source, shape.lse_stride_token = lses.stride()[:2]
    shape.out_stride_token, shape.out_stride_head = out.stride()[:2]
    shape.lse_out_stride_token = 0 if lse_out is None else lse_out.stride(0)
    if stream is None:
        stream = torch.cuda.current_stream(out.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    rc = lib.smla_merge(ctypes.byref(shape), _ptr(parts), _ptr(lses), _ptr(lens), _ptr(out), _ptr(lse_out),
                        ctypes.c_void_p(handle))
    if rc != OK:
        raise SmlaError(rc, "smla_merge")
    return out, lse_out


def merge(parts, lses, lens=None, stream=None, with_lse=True):
    """Allocates the outputs on parts' device and calls :func:`smla_merge`."""
    S, T, H, _ = parts.shape
    out = torch.empty((T, H, LATENT), dtype=torch.bfloat16, device=parts.device)
    lse_out = torch.empty((T, H), dtype=torch.float32, device=parts.device) if with_lse else None
    return smla_merge(parts, lses, lens, out, lse_out, stream=stream)


def smla_mxfp4_q_quant(q: torch.Tensor, weights: torch.Tensor, weight_scale: float, q_packed: torch.Tensor,
                       q_scale: torch.Tensor, w_out: torch.Tensor, stream=None):
    """MXFP4 quantisation of the indexer query through the C ABI (see
    ``smla_mxfp4_q_quant`` in smla.h). q: bfloat16 or float32 [T, H, 128],
    values contiguous; weights float32 [T, H]; q_packed uint8 [T, P, 64];
    q_scale int32 [T, P]; w_out float32 [T, P]."""
    lib = load()
    T, H, D = q.shape
    P = q_packed.shape[1]
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("mxfp4: q must be bfloat16 or float32")
    if tuple(weights.shape) != (T, H) or tuple(q_packed.shape) != (T, P, D // 2) or tuple(q_scale.shape) != (T, P) \
            or tuple(w_out.shape) != (T, P):
        raise ValueError("mxfp4: shapes")
    if q.stride(2) != 1 or (H > 1 and weights.stride(1) != 1) or q_packed.stride(2) != 1 \
            or (P > 1 and (q_packed.stride(1) != D // 2 or q_scale.stride(1) != 1 or w_out.stride(1) != 1)):
        raise ValueError("mxfp4: inner dimensions must be contiguous")
    shape = SmlaMxfp4Shape()
    shape.tokens, shape.heads, shape.padded_heads, shape.head_dim = T, H, P, D
    shape.q_dtype = DTYPE_F32 if q.dtype == torch.float32 else DTYPE_BF16
    shape.reserved = 0
    shape.q_stride_token, shape.q_stride_head = q.stride(0), q.stride(1)
    shape.w_stride_token = weights.stride(0)
    shape.packed_stride_token = q_packed.stride(0)
    shape.scale_stride_token = q_scale.stride(0)
    shape.w_out_stride_token = w_out.stride(0)
    if stream is None:
        stream = torch.cuda.current_stream(q_packed.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    rc = lib.smla_mxfp4_q_quant(ctypes.byref(shape), _ptr(q), _ptr(weights), float(weight_scale), _ptr(q_packed),
                                _ptr(q_scale), _ptr(w_out), ctypes.c_void_p(handle))
    if rc != OK:
        raise SmlaError(rc, "smla_mxfp4_q_quant")
    return q_packed, q_scale, w_out


def mxfp4_q_quant(q, weights, weight_scale: float, padded_heads: int | None = None, stream=None):
    """Allocates the outputs on q's device and calls :func:`smla_mxfp4_q_quant`."""
    T, H, D = q.shape
    P = H if padded_heads is None else int(padded_heads)
    packed = torch.empty((T, P, D // 2), dtype=torch.uint8, device=q.device)
    scale = torch.empty((T, P), dtype=torch.int32, device=q.device)
    w_out = torch.empty((T, P), dtype=torch.float32, device=q.device)
    return smla_mxfp4_q_quant(q, weights, weight_scale, packed, scale, w_out, stream=stream)


def smla_value_gate(latent: torch.Tensor, w_uv: torch.Tensor, gate: torch.Tensor, lens: torch.Tensor | None,
                    out: torch.Tensor, stream=None):
    """Value projection and sigmoid gate through the C ABI (see
    ``smla_value_gate`` in smla.h). latent: bfloat16 [T, H, 512], latents
    contiguous; w_uv: bfloat16 [H, 512, 128] contiguous; gate and out:
    bfloat16 [T, H*128], rows contiguous; lens: int32 [T] or None."""
    lib = load()
    T, H, J = latent.shape
    if latent.dtype != torch.bfloat16 or w_uv.dtype != torch.bfloat16 or gate.dtype != torch.bfloat16 \
            or out.dtype != torch.bfloat16:
        raise ValueError("value_gate: latent, w_uv, gate and out must be bfloat16")
    if J != LATENT or tuple(w_uv.shape) != (H, LATENT, VALUE_DIM) or tuple(gate.shape) != (T, H * VALUE_DIM) \
            or tuple(out.shape) != (T, H * VALUE_DIM):
        raise ValueError("value_gate: shapes")
    if not w_uv.is_contiguous() or latent.stride(2) != 1 or gate.stride(1) != 1 or out.stride(1) != 1:
        raise ValueError("value_gate: inner dimensions must be contiguous")
    if lens is not None and (lens.dtype != torch.int32 or tuple(lens.shape) != (T,) or lens.stride(0) != 1):
        raise ValueError("value_gate: lens must be contiguous int32 [T]")
    shape = SmlaValueShape()
    shape.tokens, shape.heads = T, H
    shape.latent_stride_token, shape.latent_stride_head = latent.stride(0), latent.stride(1)
    shape.gate_stride_token, shape.out_stride_token = gate.stride(0), out.stride(0)
    if stream is None:
        stream = torch.cuda.current_stream(out.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    rc = lib.smla_value_gate(ctypes.byref(shape), _ptr(latent), _ptr(w_uv), _ptr(gate),
                             None if lens is None else _ptr(lens), _ptr(out), ctypes.c_void_p(handle))
    if rc != OK:
        raise SmlaError(rc, "smla_value_gate")
    return out


def value_gate(latent, w_uv, gate, lens=None, stream=None):
    """Allocates the output on latent's device and calls :func:`smla_value_gate`."""
    T, H, _ = latent.shape
    out = torch.empty((T, H * VALUE_DIM), dtype=torch.bfloat16, device=latent.device)
    return smla_value_gate(latent, w_uv, gate, lens, out, stream=stream)


def smla_merge_value(parts: torch.Tensor, lses: torch.Tensor, lens: torch.Tensor | None, w_uv: torch.Tensor,
                     gate: torch.Tensor, out: torch.Tensor, stream=None):
    """The LSE merge, the W_UV projection and the gate in one pass through the
    C ABI (see ``smla_merge_value`` in smla.h). parts: bfloat16 [S, T, H, 512],
    latents contiguous; lses: float32 [S, T, H], heads contiguous; lens: int32
    [T] or None; w_uv: bfloat16 [H, 512, 128] contiguous; gate and out:
    bfloat16 [T, H*128], rows contiguous."""
    lib = load()
    S, T, H, J = parts.shape
    if J != LATENT or tuple(lses.shape) != (S, T, H):
        raise ValueError("merge_value: parts [S, T, H, 512], lses [S, T, H]")
    if parts.dtype != torch.bfloat16 or lses.dtype != torch.float32 or w_uv.dtype != torch.bfloat16 \
            or gate.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise ValueError("merge_value: dtypes")
    if tuple(w_uv.shape) != (H, LATENT, VALUE_DIM) or tuple(gate.shape) != (T, H * VALUE_DIM) \
            or tuple(out.shape) != (T, H * VALUE_DIM):
        raise ValueError("merge_value: shapes")
    if parts.stride(3) != 1 or (H > 1 and lses.stride(2) != 1) or not w_uv.is_contiguous() \
            or gate.stride(1) != 1 or out.stride(1) != 1:
        raise ValueError("merge_value: inner dimensions must be contiguous")
    if lens is not None and (lens.dtype != torch.int32 or tuple(lens.shape) != (T,) or lens.stride(0) != 1):
        raise ValueError("merge_value: lens must be contiguous int32 [T]")
    shape = SmlaMergeValueShape()
    shape.sources, shape.tokens, shape.heads, shape.reserved = S, T, H, 0
    shape.part_stride_source, shape.part_stride_token, shape.part_stride_head = parts.stride()[:3]
    shape.lse_stride_source, shape.lse_stride_token = lses.stride()[:2]
    shape.gate_stride_token, shape.out_stride_token = gate.stride(0), out.stride(0)
    if stream is None:
        stream = torch.cuda.current_stream(out.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    rc = lib.smla_merge_value(ctypes.byref(shape), _ptr(parts), _ptr(lses), _ptr(lens), _ptr(w_uv), _ptr(gate),
                              _ptr(out), ctypes.c_void_p(handle))
    if rc != OK:
        raise SmlaError(rc, "smla_merge_value")
    return out


def merge_value(parts, lses, w_uv, gate, lens=None, stream=None):
    """Allocates the output on parts' device and calls :func:`smla_merge_value`."""
    _, T, H, _ = parts.shape
    out = torch.empty((T, H * VALUE_DIM), dtype=torch.bfloat16, device=parts.device)
    return smla_merge_value(parts, lses, lens, w_uv, gate, out, stream=stream)
