"""The C-ABI library builds, loads and exports every symbol include/tq.h declares.

No compute call is made here (no GPU needed).
"""
import os
import re

import pytest

from rotated_codebook_kv_gb300 import build, native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return native.load()


def test_header_declares_the_boundary():
    syms = _declared_symbols()
    for s in ("tq_init", "tq_compress_kv", "tq_dequant_kv", "tq_decode_attention"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    for s in _declared_symbols():
        assert hasattr(lib, s), s
    assert set(_declared_symbols()) <= set(native.SIGNATURES)


def test_invalid_arguments_rejected_without_gpu(lib):
    # argument validation happens on the host before any CUDA call
    with pytest.raises(native.TQError) as e:
        native.tq_init(96, 3, 4, 32, 0)
    assert e.value.status == native.TQ_ERR_UNSUPPORTED
    assert "head_dim" in native.tq_last_error()
    with pytest.raises(native.TQError) as e:
        native.tq_init(128, 5, 4, 32, 0)
    assert e.value.status == native.TQ_ERR_UNSUPPORTED
    with pytest.raises(native.TQError) as e:
        native.tq_init(128, 3, 4, 48, 0)
    assert e.value.status == native.TQ_ERR_UNSUPPORTED
    with pytest.raises(native.TQError) as e:
        native.tq_compress_kv(None, 0, 0, 1, 1, 128, 128, 0, 0, 0, 16, 1, None)
    assert e.value.status == native.TQ_ERR_INVALID_ARG
    with pytest.raises(native.TQError) as e:  # an option flag the library does not know
        native.tq_init_ex(128, 3, 4, 32, 0, 0x10)
    assert e.value.status == native.TQ_ERR_UNSUPPORTED and "flags" in native.tq_last_error()
    assert native.tq_decode_workspace_bytes(None, 1, 1, 1) == 0


def test_every_entry_point_rejects_a_null_handle(lib):
    # host-side checks only: no CUDA call is reached with a NULL handle
    calls = {
        "tq_cache_layout": lambda: native.tq_cache_layout(None, 16),
        "tq_dequant_kv": lambda: native.tq_dequant_kv(None, 0, 0, 16, 1, 1, 0, 1, 0, 0, None),
        "tq_decode_attention": lambda: native.tq_decode_attention(None, 0, 0, 0, 0, 0, 1, 1, 1, 16, 1, 1, 1.0, 1, 0, 0,
                                                                  0, None),
        "tq_decode_attention_static": lambda: native.tq_decode_attention_static(None, 0, 0, 0, 0, 0, 1, 1, 1, 16, 1,
                                                                                1, 1.0, 1, 0, None),
        "tq_prefill_attention": lambda: native.tq_prefill_attention(None, 0, 0, 0, 0, 0, 1, 1, 1, 1, 16, 1, 1, 1.0,
                                                                    1, 0, 0, 0, None),
        "tq_decode_attention_bf16": lambda: native.tq_decode_attention_bf16(None, 0, 0, 0, 0, 0, 1, 1, 1, 16, 1, 1,
                                                                            1.0, 1, 0, 0, 0, None),
        "tq_set_wait_limit": lambda: native.tq_set_wait_limit(None, 5),
        "tq_get_status": lambda: native.tq_get_status(None, None),
        "tq_export_params": lambda: native.tq_export_params(None, None, None, None, None),
    }
    for name, call in calls.items():
        with pytest.raises(native.TQError) as e:
            call()
        assert e.value.status == native.TQ_ERR_INVALID_ARG, name
        assert "NULL" in native.tq_last_error(), name
    native.tq_destroy(None)  # a NULL handle is a no-op
    assert native.tq_decode_splits(None, 1, 1, 1, 16) == 1
