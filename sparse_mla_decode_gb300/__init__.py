"""Sparse MLA decode attention for GB300 (sm_103a).

The compute lives in ``libsmla.so`` (hand-written CUDA, C ABI in
``include/smla.h``); :mod:`sparse_mla_decode_gb300.smla` is its thin Python
binding and :mod:`sparse_mla_decode_gb300.workloads` draws seeded inputs.
"""

from .smla import (  # noqa: F401
    SmlaError,
    decode,
    decode_ds_mla,
    load,
    make_shape,
    merge,
    merge_value,
    mxfp4_q_quant,
    smla_decode,
    smla_decode_ds_mla,
    smla_ds_mla_head_tile,
    smla_device_error,
    smla_read_device_error,
    smla_selftest_bounded_wait,
    smla_merge,
    smla_merge_value,
    smla_mxfp4_q_quant,
    smla_plan_for,
    smla_value_gate,
    smla_version,
    value_gate,
)
