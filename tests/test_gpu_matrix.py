"""GPU parity over the whole supported parameter set, plus special inputs.

tq_init accepts head_dim {128, 256} x k_bits {2, 3, 4} x v_bits {2, 3, 4} x
group {32, 64, 128} x page {16, 32}, and decode accepts any whole GQA ratio
G = Hq / Hkv in 1..8.  Every (head_dim, k_bits, v_bits) pair runs here, with
group, page size and G cycled so that each value of each appears for both head
dims.  Every case compresses (records checked against the oracle), decodes
(outputs checked element by element against the oracle on the GPU-written
cache) and checks the raw fp32 decode output, read from the workspace before
its bf16 rounding, against the plain 2e-3 tolerance.  Special inputs ride
along in every case: exact-zero key rows, value groups that are constant
(scale 0), and all-zero value rows.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle as O
from parity import DECODE_ATOL, check_decode, check_key_value_records, read_records
from rotated_codebook_kv_gb300 import Codec
from rotated_codebook_kv_gb300 import workloads as W

DEV = "cuda"

GROUPS = (32, 64, 128)
PAGES = (16, 32)
GQA = (1, 3, 8, 2, 5)


def _cases():
    out = []
    for i, (d, kb, vb) in enumerate(itertools.product((128, 256), (2, 3, 4), (2, 3, 4))):
        j = i % 9
        out.append(dict(d=d, kb=kb, vb=vb, g=GROUPS[j % 3], P=PAGES[(j // 3 + j) % 2], G=GQA[j % len(GQA)]))
    return out


CASES = _cases()


def _ids(c):
    return f"d{c['d']}-k{c['kb']}v{c['vb']}-g{c['g']}-P{c['P']}-G{c['G']}"


def test_matrix_covers_every_value():
    for d in (128, 256):
        sub = [c for c in CASES if c["d"] == d]
        assert {c["g"] for c in sub} == set(GROUPS)
        assert {c["P"] for c in sub} == set(PAGES)
        assert {(c["kb"], c["vb"]) for c in sub} == set(itertools.product((2, 3, 4), (2, 3, 4)))
    assert {1, 3, 8} <= {c["G"] for c in CASES}


def _special_inputs(b, g):
    """Zero key rows, constant value groups and zero value rows on fixed tokens."""
    k, v = b.k.float(), b.v.float()
    T = k.shape[0]
    k[3] = 0.0                      # exact-zero key rows (every head)
    k[T // 2, 0] = 0.0
    v[5, :, :g] = 1.5               # a constant value group on every head
    if 2 * g <= v.shape[-1]:
        v[7, 0, g:2 * g] = -0.25
    v[11] = 0.0                     # all-zero value rows
    b.k, b.v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    return b


@pytest.mark.gpu
@pytest.mark.parametrize("c", CASES, ids=[_ids(c) for c in CASES])
def test_parameter_matrix(c):
    Hkv = 2
    w = W.Workload("matrix", c["d"], c["kb"], c["vb"], c["g"], c["P"], num_kv_heads=Hkv,
                   num_q_heads=Hkv * c["G"], batch=3, seq_len_range=(150, 420),
                   seed=c["d"] + 10 * c["kb"] + c["vb"])
    b = _special_inputs(W.generate(w, device="cpu"), c["g"])
    b = W.Batch(**{f: (getattr(b, f).to(DEV) if isinstance(getattr(b, f), torch.Tensor) else getattr(b, f))
                   for f in b.__dataclass_fields__})
    seed = w.codec_seed()
    codec = Codec(c["d"], c["kb"], c["vb"], c["g"], seed)
    ora = O.Oracle(c["d"], c["kb"], c["vb"], c["g"], seed)
    kc, vc = codec.alloc_cache(b.num_blocks, Hkv, c["P"], fill=0xA5)
    codec.compress_kv(b.k, b.v, b.slot_mapping, kc, vc, c["P"], b.num_blocks)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    # records of every written token against the oracle
    sm = b.slot_mapping.cpu().numpy()
    tok = np.nonzero(sm >= 0)[0]
    kc_np, vc_np = kc.cpu().numpy(), vc.cpu().numpy()
    rec = read_records(kc_np, vc_np, ora.geometry(c["P"]), c["d"], c["kb"], c["vb"], c["g"], c["P"], Hkv, sm[tok])
    check_key_value_records(ora, W.as_u16(b.k).reshape(-1, c["d"]), W.as_u16(b.v).reshape(-1, c["d"]), rec)
    # zero keys are all-zero records; constant groups have scale 0
    assert not rec["k_code"][3].any() and not rec["k_norm"][3].any()
    assert np.all(rec["v_meta"][5, :, 0, 0] == 0)
    # decode: bf16 outputs and the raw fp32 outputs in the workspace
    splits = codec.decode_splits(w.batch, Hkv, b.block_table.shape[1], c["P"])
    ws = codec.workspace(w.batch, w.num_q_heads, splits)
    out = codec.decode_attention(b.q, kc, vc, b.block_table, b.seq_lens, Hkv, c["P"], b.num_blocks, b.sm_scale,
                                 splits=splits, workspace=ws)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    ref = ora.decode(W.as_u16(b.q), kc_np, vc_np, b.block_table.cpu().numpy(), b.seq_lens.cpu().numpy(), Hkv,
                     c["P"], b.sm_scale, mode=1)
    check_decode(W.as_u16(out), ref)
    n = w.batch * w.num_q_heads * c["d"]
    raw = ws[: 4 * n].view(torch.float32).reshape(ref.shape).cpu().numpy().astype(np.float64)
    err = np.abs(raw - ref)
    assert err.max() <= DECODE_ATOL, f"raw fp32 decode error {err.max():.3e}"
