"""ctypes binding of ``libtq.so`` (the C ABI in ``include/tq.h``).

Argument marshalling only: every function has the C name and forwards plain
integers / device pointers.  The library is loaded from the package's
``_lib`` folder (built in-tree by ``build.py``); if it is missing the import
of this module raises -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA, TQ_ERR_OOM = range(5)
TQ_ROTATION_DENSE, TQ_ROTATION_HADAMARD, TQ_VALUES_MSE = 0, 1, 2
TQ_DEVERR_SLOT_RANGE, TQ_DEVERR_BLOCK_RANGE, TQ_DEVERR_SEQ_RANGE, TQ_DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8
TQ_DEFAULT_WAIT_LIMIT = 2000000000

# Every symbol include/tq.h declares, with (restype, argtypes).
_c = ctypes
_vp, _i32, _i64, _u64, _sz, _f32 = _c.c_void_p, _c.c_int, _c.c_int64, _c.c_uint64, _c.c_size_t, _c.c_float
SIGNATURES = {
    "tq_init": (_i32, [_i32, _i32, _i32, _i32, _u64, _c.POINTER(_vp)]),
    "tq_init_ex": (_i32, [_i32, _i32, _i32, _i32, _u64, _c.c_uint, _c.POINTER(_vp)]),
    "tq_destroy": (_i32, [_vp]),
    "tq_cache_layout": (_i32, [_vp, _i32, _c.POINTER(_sz), _c.POINTER(_sz)]),
    "tq_compress_kv": (_i32, [_vp, _vp, _vp, _i64, _i32, _i64, _i64, _vp, _vp, _vp, _i32, _i64, _vp]),
    "tq_dequant_kv": (_i32, [_vp, _vp, _vp, _i32, _i64, _i32, _vp, _i64, _vp, _vp, _vp]),
    "tq_decode_splits": (_i32, [_vp, _i32, _i32, _i32, _i32]),
    "tq_decode_workspace_bytes": (_sz, [_vp, _i32, _i32, _i32]),
    "tq_decode_attention": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _f32, _i32,
                                   _vp, _sz, _vp, _vp]),
    "tq_prefill_queries_per_cta": (_i32, [_vp, _i32, _i32]),
    "tq_prefill_splits": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _i32]),
    "tq_prefill_attention": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i64, _f32,
                                    _i32, _vp, _sz, _vp, _vp]),
    "tq_decode_attention_bf16": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _f32,
                                        _i32, _vp, _sz, _vp, _vp]),
    "tq_decode_attention_static": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _f32,
                                          _i32, _vp, _vp]),
    "tq_set_wait_limit": (_i32, [_vp, _i64]),
    "tq_get_status": (_i32, [_vp, _c.POINTER(_c.c_uint32), _vp]),
    "tq_export_params": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "tq_last_error": (_c.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


class TQError(RuntimeError):
    def __init__(self, func: str, status: int, message: str):
        super().__init__(f"{func} failed with status {status}: {message}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libtq.so (building it first if it is missing or stale and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and _build.is_stale():
            _build.build()
        if not os.path.exists(path):
            raise ImportError(f"libtq.so not found at {path}; run rotated_codebook_kv_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(name: str, status: int):
    if status != TQ_OK:
        raise TQError(name, status, load().tq_last_error().decode())


def tq_last_error() -> str:
    return load().tq_last_error().decode()


def tq_init(head_dim: int, k_bits: int, v_bits: int, group: int, seed: int) -> int:
    h = _vp()
    _check("tq_init", load().tq_init(head_dim, k_bits, v_bits, group, seed, ctypes.byref(h)))
    return h.value


def tq_init_ex(head_dim: int, k_bits: int, v_bits: int, group: int, seed: int, flags: int) -> int:
    h = _vp()
    _check("tq_init_ex", load().tq_init_ex(head_dim, k_bits, v_bits, group, seed, flags, ctypes.byref(h)))
    return h.value


def tq_destroy(h: int) -> None:
    _check("tq_destroy", load().tq_destroy(h))


def tq_cache_layout(h: int, page_size: int):
    kb, vb = _sz(), _sz()
    _check("tq_cache_layout", load().tq_cache_layout(h, page_size, ctypes.byref(kb), ctypes.byref(vb)))
    return kb.value, vb.value


def tq_compress_kv(h, k, v, T, num_kv_heads, k_stride_tok, v_stride_tok, slot_mapping, k_cache, v_cache,
                   page_size, num_blocks, stream) -> None:
    _check("tq_compress_kv", load().tq_compress_kv(h, k, v, T, num_kv_heads, k_stride_tok, v_stride_tok,
                                                   slot_mapping, k_cache, v_cache, page_size, num_blocks, stream))


def tq_dequant_kv(h, k_cache, v_cache, page_size, num_blocks, num_kv_heads, slots, T, k_out, v_out, stream) -> None:
    _check("tq_dequant_kv", load().tq_dequant_kv(h, k_cache, v_cache, page_size, num_blocks, num_kv_heads, slots, T,
                                                 k_out, v_out, stream))


def tq_decode_splits(h, batch, num_kv_heads, max_blocks_per_seq, page_size) -> int:
    return load().tq_decode_splits(h, batch, num_kv_heads, max_blocks_per_seq, page_size)


def tq_decode_workspace_bytes(h, batch, num_q_heads, splits) -> int:
    return load().tq_decode_workspace_bytes(h, batch, num_q_heads, splits)


def tq_decode_attention(h, q, k_cache, v_cache, block_table, seq_lens, batch, num_q_heads, num_kv_heads, page_size,
                        max_blocks_per_seq, num_blocks, sm_scale, splits, workspace, ws_bytes, out, stream) -> None:
    _check("tq_decode_attention", load().tq_decode_attention(
        h, q, k_cache, v_cache, block_table, seq_lens, batch, num_q_heads, num_kv_heads, page_size,
        max_blocks_per_seq, num_blocks, sm_scale, splits, workspace, ws_bytes, out, stream))


def tq_prefill_queries_per_cta(h, num_q_heads, num_kv_heads) -> int:
    return load().tq_prefill_queries_per_cta(h, num_q_heads, num_kv_heads)


def tq_prefill_splits(h, batch, q_tokens, num_q_heads, num_kv_heads, max_blocks_per_seq, page_size) -> int:
    return load().tq_prefill_splits(h, batch, q_tokens, num_q_heads, num_kv_heads, max_blocks_per_seq, page_size)


def tq_prefill_attention(h, q, k_cache, v_cache, block_table, seq_lens, batch, q_tokens, num_q_heads, num_kv_heads,
                         page_size, max_blocks_per_seq, num_blocks, sm_scale, splits, workspace, ws_bytes, out,
                         stream) -> None:
    _check("tq_prefill_attention", load().tq_prefill_attention(
        h, q, k_cache, v_cache, block_table, seq_lens, batch, q_tokens, num_q_heads, num_kv_heads, page_size,
        max_blocks_per_seq, num_blocks, sm_scale, splits, workspace, ws_bytes, out, stream))


def tq_decode_attention_bf16(h, q, k_pool, v_pool, block_table, seq_lens, batch, num_q_heads, num_kv_heads,
                             page_size, max_blocks_per_seq, num_blocks, sm_scale, splits, workspace, ws_bytes, out,
                             stream) -> None:
    _check("tq_decode_attention_bf16", load().tq_decode_attention_bf16(
        h, q, k_pool, v_pool, block_table, seq_lens, batch, num_q_heads, num_kv_heads, page_size,
        max_blocks_per_seq, num_blocks, sm_scale, splits, workspace, ws_bytes, out, stream))


def tq_decode_attention_static(h, q, k_cache, v_cache, block_table, seq_lens, batch, num_q_heads, num_kv_heads,
                               page_size, max_blocks_per_seq, num_blocks, sm_scale, splits, out, stream) -> None:
    _check("tq_decode_attention_static", load().tq_decode_attention_static(
        h, q, k_cache, v_cache, block_table, seq_lens, batch, num_q_heads, num_kv_heads, page_size,
        max_blocks_per_seq, num_blocks, sm_scale, splits, out, stream))


def tq_set_wait_limit(h, cycles: int) -> None:
    _check("tq_set_wait_limit", load().tq_set_wait_limit(h, cycles))


def tq_get_status(h, stream) -> int:
    bits = ctypes.c_uint32()
    _check("tq_get_status", load().tq_get_status(h, ctypes.byref(bits), stream))
    return bits.value


def tq_export_params(h, Pi, S, centroids, thresholds) -> None:
    _check("tq_export_params", load().tq_export_params(h, Pi, S, centroids, thresholds))
