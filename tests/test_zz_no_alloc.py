"""The allocation-free decode entry point against the workspace entry point.

tq_decode_attention_static serves callers that cannot allocate device memory:
it keeps its scratch in a static device array.  Through the C ABI, two calls in
a row must give the same outputs as tq_decode_attention with a caller-provided
workspace (within the decode tolerance the other tests use), and a call whose
scratch would not fit must be refused before any launch.  This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity import DECODE_ATOL
from rotated_codebook_kv_gb300 import Codec, native
from rotated_codebook_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _case():
    w = W.scaled(W.paged_decode(), batch=6, seq_len_range=(200, 900))
    b = W.generate(w, device="cuda")
    codec = Codec(w.head_dim, w.k_bits, w.v_bits, w.group, w.codec_seed())
    kc, vc = codec.alloc_cache(b.num_blocks, w.num_kv_heads, w.page_size)
    codec.compress_kv(b.k, b.v, b.slot_mapping, kc, vc, w.page_size, b.num_blocks)
    return w, b, codec, kc, vc


def _args(w, b, kc, vc):
    return (b.q.data_ptr(), kc.data_ptr(), vc.data_ptr(), b.block_table.data_ptr(), b.seq_lens.data_ptr(),
            w.batch, w.num_q_heads, w.num_kv_heads, w.page_size, b.block_table.shape[1], b.num_blocks, b.sm_scale)


def test_static_scratch_matches_workspace_entry_point():
    w, b, codec, kc, vc = _case()
    stream = torch.cuda.current_stream().cuda_stream
    splits = native.tq_decode_splits(codec.handle, w.batch, w.num_kv_heads, b.block_table.shape[1], w.page_size)
    ws_bytes = native.tq_decode_workspace_bytes(codec.handle, w.batch, w.num_q_heads, splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(b.q)
    native.tq_decode_attention(codec.handle, *_args(w, b, kc, vc), splits, ws.data_ptr(), ws_bytes, ref.data_ptr(),
                               stream)
    for _ in range(2):  # the second call reuses the array's previous contents
        out = torch.full_like(b.q, float("nan"))
        native.tq_decode_attention_static(codec.handle, *_args(w, b, kc, vc), splits, out.data_ptr(), stream)
        torch.cuda.synchronize()
        assert native.tq_get_status(codec.handle, stream) == 0
        g = O.bf16_to_double(W.as_u16(out))
        r = O.bf16_to_double(W.as_u16(ref))
        assert np.all(np.isfinite(g))
        assert np.abs(g - r).max() <= DECODE_ATOL


def test_static_scratch_rejects_oversized_calls():
    w, b, codec, kc, vc = _case()
    stream = torch.cuda.current_stream().cuda_stream
    big_batch = 4096  # 4096 x 32 heads x 64 splits of partials cannot fit 16 MiB
    with pytest.raises(native.TQError) as e:
        native.tq_decode_attention_static(codec.handle, b.q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                          b.block_table.data_ptr(), b.seq_lens.data_ptr(), big_batch, w.num_q_heads,
                                          w.num_kv_heads, w.page_size, b.block_table.shape[1], b.num_blocks,
                                          b.sm_scale, 64, b.q.data_ptr(), stream)
    assert e.value.status == native.TQ_ERR_UNSUPPORTED
    assert "static array" in native.tq_last_error()
