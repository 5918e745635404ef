"""GPU parity of chunked prefill over the compressed cache.

tq_prefill_attention (the last q_tokens positions of every sequence attend
causally to the compressed cache, their own keys and values included) against
the oracle's causal attention, element by element (2e-3 + half a bf16 ulp).
head_dim 128 runs the tensor-memory kernel (128 columns per CTA, 64-token
tiles): GQA ratios 1, 2, 3, 4 and 8, chunks that do not fill the last CTA,
sequences shorter than the chunk and sequences of many tiles, both page sizes,
with and without QJL, every value width, several split counts, a key scale that
grows along the sequence (the lazy rescale of O), timeouts, bad block ids and the
full-size paged workload (sampled sequences).  head_dim 256 runs the decode's
split-K kernel (one to eight query tokens per CTA).  The last query token of a
sequence is checked against the decode of the whole sequence.
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
    (128, 3, 3, 32, 16, 4, [700, 65], 70),    # three CTAs of 32 query tokens, the last holding 6
    (128, 2, 4, 64, 32, 1, [260, 1500], 130), # G 1: 128 query tokens per CTA; 24 tiles of 64 tokens
    (128, 4, 2, 128, 16, 3, [333, 90], 50),   # G 3: 42 query tokens (126 columns) per CTA
    (128, 4, 3, 32, 32, 8, [1100, 5], 17),    # G 8: 16 query tokens per CTA; a 5-token sequence
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
    # head_dim 128: 128 (token, head) columns per CTA; 256: 8
    codec = Codec(128, 4, 4, 32, 0)
    assert [native.tq_prefill_queries_per_cta(codec.handle, 2 * G, 2) for G in (1, 2, 3, 4, 8)] == [128, 64, 42, 32, 16]
    wide = Codec(256, 4, 4, 64, 0)
    assert [native.tq_prefill_queries_per_cta(wide.handle, 2 * G, 2) for G in (1, 2, 3, 4, 8)] == [8, 4, 2, 2, 1]


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


def _prefill_setup(d, kb, vb, g, P, G, lens, Tq, Hkv=2, seed=0, values="group"):
    w, b, q = _case(d, kb, vb, g, P, G, lens, Tq, Hkv=Hkv, seed=seed)
    codec = Codec(d, kb, vb, g, w.codec_seed(), values=values)
    ora = O.Oracle(d, kb, vb, g, w.codec_seed(), values=values)
    return w, b, q, codec, ora


def test_prefill_lazy_rescale_with_growing_scores():
    """Keys scaled by 1, 4 and 16 along the sequence: the running maximum of a column
    grows by far more than 2^8 between tiles, so the kernel rescales O in tensor
    memory several times; results still match the oracle."""
    d, kb, vb, g, P, G, Hkv = 128, 3, 4, 32, 16, 4, 2
    lens, Tq = [900], 40
    w, b, q, codec, ora = _prefill_setup(d, kb, vb, g, P, G, lens, Tq, Hkv=Hkv, seed=21)
    k = b.k.float()
    pos = torch.arange(k.shape[0])
    k *= torch.where(pos < 300, 1.0, torch.where(pos < 600, 4.0, 16.0))[:, None, None]
    b.k = k.to(torch.bfloat16)
    kc, vc = codec.alloc_cache(b.num_blocks, Hkv, P)
    codec.compress_kv(b.k.to(DEV), b.v.to(DEV), b.slot_mapping.to(DEV), kc, vc, P, b.num_blocks)
    out = codec.prefill_attention(q.to(DEV), kc, vc, b.block_table.to(DEV), b.seq_lens.to(DEV), Hkv, P,
                                  b.num_blocks, b.sm_scale, splits=1)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    ref = ora.prefill(W.as_u16(q), kc.cpu().numpy(), vc.cpu().numpy(), b.block_table.numpy(), b.seq_lens.numpy(),
                      Hkv, P, b.sm_scale)
    check_decode(W.as_u16(out), ref)


def test_prefill_wait_timeouts_report_and_recover():
    """With a wait limit of 0 every barrier wait of the tensor-memory prefill tests
    once and gives up if its phase has not completed (the first page copies have
    not): TQ_DEVERR_TIMEOUT, finite outputs, and with the default limit restored
    the same call gives the normal results again."""
    d, kb, vb, g, P, G, Hkv = 128, 3, 2, 32, 16, 4, 2
    w, b, q, codec, ora = _prefill_setup(d, kb, vb, g, P, G, [600, 200], 24, Hkv=Hkv, seed=5)
    kc, vc = codec.alloc_cache(b.num_blocks, Hkv, P)
    codec.compress_kv(b.k.to(DEV), b.v.to(DEV), b.slot_mapping.to(DEV), kc, vc, P, b.num_blocks)
    args = (q.to(DEV), kc, vc, b.block_table.to(DEV), b.seq_lens.to(DEV), Hkv, P, b.num_blocks, b.sm_scale)
    ref = codec.prefill_attention(*args)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    codec.set_wait_limit(0)
    out = codec.prefill_attention(*args)
    torch.cuda.synchronize()
    assert codec.get_status() & native.TQ_DEVERR_TIMEOUT
    assert np.all(np.isfinite(O.bf16_to_double(W.as_u16(out))))
    codec.set_wait_limit(native.TQ_DEFAULT_WAIT_LIMIT)
    again = codec.prefill_attention(*args)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    assert torch.equal(again, ref)


def test_prefill_bad_block_sets_status():
    d, kb, vb, g, P, G, Hkv = 128, 4, 4, 64, 16, 2, 2
    w, b, q, codec, ora = _prefill_setup(d, kb, vb, g, P, G, [500, 300], 16, Hkv=Hkv, seed=6)
    kc, vc = codec.alloc_cache(b.num_blocks, Hkv, P, fill=0xA5)
    codec.compress_kv(b.k.to(DEV), b.v.to(DEV), b.slot_mapping.to(DEV), kc, vc, P, b.num_blocks)
    bt = b.block_table.clone()
    bt[0, 3] = b.num_blocks + 7
    out = codec.prefill_attention(q.to(DEV), kc, vc, bt.to(DEV), b.seq_lens.to(DEV), Hkv, P, b.num_blocks,
                                  b.sm_scale)
    torch.cuda.synchronize()
    assert codec.get_status() & native.TQ_DEVERR_BLOCK_RANGE
    assert np.all(np.isfinite(O.bf16_to_double(W.as_u16(out))))


def test_prefill_full_size_paged_workload_sampled():
    """The benchmark's prefill case at full size (the paged decode workload: 32
    sequences of 1,024-8,192 tokens, 8 kv heads, G 4, page 16; a chunk of 64 query
    tokens per sequence, the split count the library picks), checked against the
    oracle on the shortest and the longest sequence."""
    w = W.paged_decode()
    b = W.generate(w, device=DEV)
    codec = Codec(w.head_dim, w.k_bits, w.v_bits, w.group, w.codec_seed())
    ora = O.Oracle(w.head_dim, w.k_bits, w.v_bits, w.group, w.codec_seed())
    kc, vc = codec.alloc_cache(b.num_blocks, w.num_kv_heads, w.page_size)
    codec.compress_kv(b.k, b.v, b.slot_mapping, kc, vc, w.page_size, b.num_blocks)
    Tq = 64
    gq = torch.Generator(device=DEV).manual_seed(5)
    q = torch.randn(w.batch, Tq, w.num_q_heads, w.head_dim, generator=gq, device=DEV).to(torch.bfloat16)
    out = codec.prefill_attention(q, kc, vc, b.block_table, b.seq_lens, w.num_kv_heads, w.page_size, b.num_blocks,
                                  b.sm_scale)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    lens = b.seq_lens.cpu().numpy()
    kc_np, vc_np = kc.cpu().numpy(), vc.cpu().numpy()
    for s in (int(np.argmin(lens)), int(np.argmax(lens))):
        ref = ora.prefill(W.as_u16(q[s:s + 1]), kc_np, vc_np, b.block_table[s:s + 1].cpu().numpy(), lens[s:s + 1],
                          w.num_kv_heads, w.page_size, b.sm_scale)
        check_decode(W.as_u16(out[s:s + 1]), ref)


@pytest.mark.parametrize("kb,vb", [(2, 2), (3, 4), (4, 3)])
def test_prefill_value_widths_and_mse_values(kb, vb):
    """Every value width through the tensor-memory kernel's value decode, with the
    group quantiser and with values coded by the rotation."""
    d, g, P, G, Hkv = 128, 32, 16, 4, 2
    for values in ("group", "mse"):
        w, b, q, codec, ora = _prefill_setup(d, kb, vb, g, P, G, [330, 129], 33, Hkv=Hkv, seed=kb * 7 + vb,
                                             values=values)
        kc, vc = codec.alloc_cache(b.num_blocks, Hkv, P, fill=0xA5)
        codec.compress_kv(b.k.to(DEV), b.v.to(DEV), b.slot_mapping.to(DEV), kc, vc, P, b.num_blocks)
        out = codec.prefill_attention(q.to(DEV), kc, vc, b.block_table.to(DEV), b.seq_lens.to(DEV), Hkv, P,
                                      b.num_blocks, b.sm_scale, splits=2)
        torch.cuda.synchronize()
        assert codec.get_status() == 0
        ref = ora.prefill(W.as_u16(q), kc.cpu().numpy(), vc.cpu().numpy(), b.block_table.numpy(),
                          b.seq_lens.numpy(), Hkv, P, b.sm_scale)
        check_decode(W.as_u16(out), ref)
