"""GPU parity of the bypass decode (plain bf16 pages through the decode skeleton).

tq_decode_attention_bf16 against the oracle's softmax attention over the same
bf16 pools, element by element (|gpu - oracle| <= 2e-3 + half a bf16 ulp), over
head dims, page sizes, GQA ratios, ragged lengths that end inside a round and
inside a page, and split counts; plus bad block ids and the wait-timeout path.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity import check_decode
from rotated_codebook_kv_gb300 import Codec, native

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(d, P, G, lens, Hkv=2, seed=0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    lens = torch.tensor(lens, dtype=torch.int32)
    npg = (lens + P - 1) // P
    nb = int(npg.sum()) + 3
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    B = len(lens)
    bt = torch.full((B, max(int(npg.max()), 1)), -1, dtype=torch.int32)
    st = 0
    for b in range(B):
        bt[b, : npg[b]] = perm[st: st + int(npg[b])]
        st += int(npg[b])
    kp = torch.randn(nb, Hkv, P, d, generator=g).to(torch.bfloat16)
    vp = torch.randn(nb, Hkv, P, d, generator=g).to(torch.bfloat16)
    q = torch.randn(B, Hkv * G, d, generator=g).to(torch.bfloat16)
    return q, kp, vp, bt, lens, nb


def _u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _run(codec, q, kp, vp, bt, lens, nb, Hkv, P, splits=0):
    out = codec.decode_attention_bf16(q.to(DEV), kp.to(DEV), vp.to(DEV), bt.to(DEV), lens.to(DEV), Hkv, P, nb,
                                      q.shape[-1] ** -0.5, splits=splits)
    torch.cuda.synchronize()
    return _u16(out.cpu())


@pytest.mark.parametrize("d,P,G,lens", [
    (128, 16, 8, [1000, 17, 640, 1, 0]),
    (128, 32, 4, [33, 95, 512]),
    (128, 16, 1, [300, 7]),
    (256, 32, 2, [700, 64, 5]),
    (256, 16, 3, [129, 250]),
])
def test_bypass_decode_matches_oracle(d, P, G, lens):
    Hkv = 2
    q, kp, vp, bt, lens_t, nb = _case(d, P, G, lens, Hkv=Hkv, seed=d + P + G)
    codec = Codec(d, 4, 4, 32, 0)
    ref = O.decode_bf16(_u16(q), _u16(kp), _u16(vp), bt.numpy(), lens_t.numpy(), Hkv, P, d ** -0.5)
    for splits in (0, 1, 3):
        out = _run(codec, q, kp, vp, bt, lens_t, nb, Hkv, P, splits)
        err = check_decode(out, ref)
        assert err < 5e-3
    assert codec.get_status() == 0


def test_bypass_bad_block_sets_status():
    d, P, Hkv = 128, 16, 2
    q, kp, vp, bt, lens, nb = _case(d, P, 4, [200, 100], Hkv=Hkv, seed=3)
    bt[0, 2] = nb + 5
    codec = Codec(d, 4, 4, 32, 0)
    out = _run(codec, q, kp, vp, bt, lens, nb, Hkv, P)
    assert codec.get_status() & native.TQ_DEVERR_BLOCK_RANGE
    assert np.all(np.isfinite(O.bf16_to_double(out)))


def test_bypass_wait_timeout_reports_and_recovers():
    d, P, Hkv = 128, 16, 2
    q, kp, vp, bt, lens, nb = _case(d, P, 2, [400, 300, 250], Hkv=Hkv, seed=4)
    codec = Codec(d, 4, 4, 32, 0)
    ref = _run(codec, q, kp, vp, bt, lens, nb, Hkv, P)
    codec.set_wait_limit(0)
    out = _run(codec, q, kp, vp, bt, lens, nb, Hkv, P)
    assert codec.get_status() & native.TQ_DEVERR_TIMEOUT
    assert np.all(np.isfinite(O.bf16_to_double(out)))
    codec.set_wait_limit(native.TQ_DEFAULT_WAIT_LIMIT)
    assert np.array_equal(_run(codec, q, kp, vp, bt, lens, nb, Hkv, P), ref)
    assert codec.get_status() == 0
