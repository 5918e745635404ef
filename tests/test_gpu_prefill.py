"""GPU parity of chunked prefill over the compressed cache.

tq_prefill_attention (the last q_tokens positions of every sequence attend
causally to the compressed cache, their own keys and values included) against
the oracle's causal attention, element by element (2e-3 + half a bf16 ulp), for
GQA ratios that give one to eight query tokens per CTA, chunks that do not fill
the last CTA, sequences shorter than the chunk, both page sizes and head dims,
with and without QJL, several split counts; and a check that decode through the
same kernel is unchanged.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity import check_decode
from rotated_codebook_kv_gb300 import Codec, native
from rotated_codebook_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(d, kb, vb, g, P, G, lens, Tq, Hkv=2, seed=0):
    w = W.Workload("prefill", d, kb, vb, g, P, num_kv_heads=Hkv, num_q_heads=Hkv * G, batch=len(lens),
                   seq_len=max(lens), seed=seed)
    b = W.generate(W.scaled(w, seq_len_range=None), device="cpu")
    # the per-sequence lengths of this case, on the same pages
    b.seq_lens = torch.tensor(lens, dtype=torch.int32)
    gq = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(len(lens), Tq, Hkv * G, d, generator=gq).to(torch.bfloat16)
    return w, b, q


@pytest.mark.parametrize("d,kb,vb,g,P,G,lens,Tq", [
    (128, 3, 2, 32, 16, 8, [300, 40], 7),     # one query token per CTA
    (128, 4, 4, 64, 16, 4, [257, 96], 5),     # two per CTA, the last CTA half full
    (128, 2, 3, 32, 32, 2, [500, 33, 3], 9),  # four per CTA; a sequence shorter than the chunk
    (128, 3, 4, 128, 16, 1, [180], 20),       # eight per CTA
    (256, 4, 4, 64, 32, 2, [400, 64], 6),
    (256, 3, 2, 32, 16, 3, [222], 4),
])
def test_prefill_matches_oracle(d, kb, vb, g, P, G, lens, Tq):
    Hkv = 2
    w, b, q = _case(d, kb, vb, g, P, G, lens, Tq, Hkv=Hkv, seed=d + kb + G)
    codec = Codec(d, kb, vb, g, w.codec_seed())
    ora = O.Oracle(d, kb, vb, g, w.codec_seed())
    kc, vc = codec.alloc_cache(b.num_blocks, Hkv, P)
    codec.compress_kv(b.k.to(DEV), b.v.to(DEV), b.slot_mapping.to(DEV), kc, vc, P, b.num_blocks)
    torch.cuda.synchronize()
    kc_np, vc_np = kc.cpu().numpy(), vc.cpu().numpy()
    ref = ora.prefill(W.as_u16(q), kc_np, vc_np, b.block_table.numpy(), b.seq_lens.numpy(), Hkv, P, b.sm_scale)
    for splits in (0, 1, 3):
        out = codec.prefill_attention(q.to(DEV), kc, vc, b.block_table.to(DEV), b.seq_lens.to(DEV), Hkv, P,
                                      b.num_blocks, b.sm_scale, splits=splits)
        torch.cuda.synchronize()
        check_decode(W.as_u16(out), ref)
    assert codec.get_status() == 0
    # the last query token of each sequence is the decode of the whole sequence
    dec = codec.decode_attention(q[:, -1].contiguous().to(DEV), kc, vc, b.block_table.to(DEV), b.seq_lens.to(DEV),
                                 Hkv, P, b.num_blocks, b.sm_scale)
    torch.cuda.synchronize()
    check_decode(W.as_u16(dec), ref[:, -1])


def test_prefill_queries_per_cta():
    codec = Codec(128, 4, 4, 32, 0)
    assert [native.tq_prefill_queries_per_cta(codec.handle, 2 * G, 2) for G in (1, 2, 3, 4, 8)] == [8, 4, 2, 2, 1]


def test_prefill_with_mse_values():
    """Prefill on a handle whose values are coded by the rotation (TQ_VALUES_MSE)."""
    d, kb, vb, P, G, Hkv = 128, 2, 3, 16, 4, 2
    w, b, q = _case(d, kb, vb, 32, P, G, [260, 70], 6, Hkv=Hkv, seed=9)
    codec = Codec(d, kb, vb, 32, w.codec_seed(), values="mse")
    ora = O.Oracle(d, kb, vb, 32, w.codec_seed(), values="mse")
    kc, vc = codec.alloc_cache(b.num_blocks, Hkv, P)
    codec.compress_kv(b.k.to(DEV), b.v.to(DEV), b.slot_mapping.to(DEV), kc, vc, P, b.num_blocks)
    out = codec.prefill_attention(q.to(DEV), kc, vc, b.block_table.to(DEV), b.seq_lens.to(DEV), Hkv, P,
                                  b.num_blocks, b.sm_scale)
    torch.cuda.synchronize()
    ref = ora.prefill(W.as_u16(q), kc.cpu().numpy(), vc.cpu().numpy(), b.block_table.numpy(), b.seq_lens.numpy(),
                      Hkv, P, b.sm_scale)
    check_decode(W.as_u16(out), ref)
    assert codec.get_status() == 0
