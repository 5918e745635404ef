"""GPU parity for values coded by the rotation and a Lloyd-Max codebook.

With TQ_VALUES_MSE the value record is codes | bf16 norm (brightcoding blog,
"What is TurboQuant-GPU?": K 2-bit + QJL with 3-bit MSE values is its 5.02x
configuration).  Compression is checked against the oracle with the same
decision windows as the keys (codes within 1e-6 of a threshold, norms one ulp at
a rounding midpoint); decode element by element against the oracle's decode on
the GPU-written cache (2e-3 + half a bf16 ulp); dequant within a bf16 ulp.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity import check_decode, check_key_value_records, read_records
from rotated_codebook_kv_gb300 import Codec, native
from rotated_codebook_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("d,kb,vb,P,G,rot", [
    (128, 2, 3, 16, 4, 0),   # the 5.02x configuration
    (128, 3, 3, 32, 8, 0),
    (128, 4, 2, 16, 2, 1),
    (256, 4, 4, 32, 2, 1),
    (256, 3, 2, 16, 3, 0),
])
def test_mse_values_compress_decode_dequant(d, kb, vb, P, G, rot):
    Hkv = 2
    w = W.Workload("vmse", d, kb, vb, 32, P, num_kv_heads=Hkv, num_q_heads=Hkv * G, batch=3,
                   seq_len_range=(150, 600), seed=11 * d + kb + vb)
    b = W.generate(w, device="cpu")
    v = b.v.float()
    v[4] = 0.0          # zero value rows: zero codes and norm
    b.v = v.to(torch.bfloat16)
    b = W.Batch(**{f: (getattr(b, f).to(DEV) if isinstance(getattr(b, f), torch.Tensor) else getattr(b, f))
                   for f in b.__dataclass_fields__})
    rotation = native.TQ_ROTATION_HADAMARD if rot else native.TQ_ROTATION_DENSE
    codec = Codec(d, kb, vb, 32, w.codec_seed(), rotation=rotation, values="mse")
    ora = O.Oracle(d, kb, vb, 32, w.codec_seed(), rotation=rot, values="mse")
    kpb, vpb = codec.cache_layout(P)
    assert vpb == P * (d * vb // 8 + 2)
    kc, vc = codec.alloc_cache(b.num_blocks, Hkv, P, fill=0xA5)
    codec.compress_kv(b.k, b.v, b.slot_mapping, kc, vc, P, b.num_blocks)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    sm = b.slot_mapping.cpu().numpy()
    kc_np, vc_np = kc.cpu().numpy(), vc.cpu().numpy()
    rec = read_records(kc_np, vc_np, ora.geometry(P), d, kb, vb, 32, P, Hkv, sm, vmse=True)
    check_key_value_records(ora, W.as_u16(b.k).reshape(-1, d), W.as_u16(b.v).reshape(-1, d), rec)
    assert not rec["v_code"][4].any() and not rec["v_norm"][4].any()
    out = codec.decode_attention(b.q, kc, vc, b.block_table, b.seq_lens, Hkv, P, b.num_blocks, b.sm_scale)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    ref = ora.decode(W.as_u16(b.q), kc_np, vc_np, b.block_table.cpu().numpy(), b.seq_lens.cpu().numpy(), Hkv, P,
                     b.sm_scale, mode=1)
    check_decode(W.as_u16(out), ref)
    slots = b.slot_mapping[::5].contiguous()
    ko, vo = codec.dequant_kv(kc, vc, P, b.num_blocks, Hkv, slots)
    torch.cuda.synchronize()
    _, rv = ora.dequant_slots(kc_np, vc_np, P, Hkv, slots.cpu().numpy())
    gv = O.bf16_to_double(W.as_u16(vo))
    ax = np.abs(rv)
    ulp = 2.0 ** (np.floor(np.log2(np.where(ax > 0, ax, 1.0))) - 7)
    assert np.all(np.abs(gv - rv) <= ulp + 1e-5)
