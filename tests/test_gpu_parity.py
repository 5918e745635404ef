"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Small cases run the oracle on every row / output; the full-size workloads run
in the same launch configuration the benchmark times and are checked on
sampled rows and sampled (sequence, kv head) outputs.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity import check_decode, check_key_value_records, read_records
from rotated_codebook_kv_gb300 import Codec
from rotated_codebook_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _codec_pair(w, layer=0):
    seed = w.codec_seed(layer)
    return (Codec(w.head_dim, w.k_bits, w.v_bits, w.group, seed),
            O.Oracle(w.head_dim, w.k_bits, w.v_bits, w.group, seed))


def _compress(codec, w, b, fill=0xA5):
    kc, vc = codec.alloc_cache(b.num_blocks, w.num_kv_heads, w.page_size, fill=fill)
    codec.compress_kv(b.k, b.v, b.slot_mapping, kc, vc, w.page_size, b.num_blocks)
    torch.cuda.synchronize()
    return kc, vc


def _rows(t):  # [T, H, d] bf16 tensor -> [T*H, d] uint16
    return W.as_u16(t).reshape(-1, t.shape[-1])


def _check_rows(ora, w, b, kc, vc, token_idx=None):
    """Compare the records of tokens `token_idx` (all heads) with the oracle."""
    geo = ora.geometry(w.page_size)
    sm = b.slot_mapping.cpu().numpy()
    if token_idx is None:
        token_idx = np.nonzero(sm >= 0)[0]
    token_idx = np.asarray(token_idx)
    slots = sm[token_idx]
    rec = read_records(kc.cpu().numpy(), vc.cpu().numpy(), geo, w.head_dim, w.k_bits, w.v_bits, w.group,
                       w.page_size, w.num_kv_heads, slots)
    tk = torch.as_tensor(token_idx, device=b.k.device)
    k_rows = _rows(b.k[tk])
    v_rows = _rows(b.v[tk])
    return check_key_value_records(ora, k_rows, v_rows, rec)


def _decode_gpu(codec, w, b, kc, vc, splits=0):
    out = codec.decode_attention(b.q, kc, vc, b.block_table, b.seq_lens, w.num_kv_heads, w.page_size,
                                 b.num_blocks, b.sm_scale, splits=splits)
    torch.cuda.synchronize()
    return W.as_u16(out)


def _decode_oracle(ora, w, b, kc_np, vc_np, jobs=None):
    return ora.decode(W.as_u16(b.q), kc_np, vc_np, b.block_table.cpu().numpy(), b.seq_lens.cpu().numpy(),
                      w.num_kv_heads, w.page_size, b.sm_scale, mode=1, jobs=jobs)


def _rows_of_jobs(w, jobs):
    G = w.num_q_heads // w.num_kv_heads
    return [(bb, kvh * G + g) for bb, kvh in jobs for g in range(G)]


# --------------------------------------------------------------------------- #
# Parameters                                                                    #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("d,kb,seed", [(128, 3, 0), (256, 4, 5), (128, 2, 7)])
def test_parameter_tables_match_oracle(d, kb, seed):
    lib = Codec(d, kb, 4, 32, seed).export_params()
    ref = O.Oracle(d, kb, 4, 32, seed).params()
    for name in ("Pi", "S", "centroids", "thresholds"):
        a = lib[name].astype(np.float64)
        r = ref[name]
        # the library rounds its double tables to fp32 once
        assert np.all(np.abs(a - r) <= np.abs(r) * 2.0 ** -24 + 1e-13), name


# --------------------------------------------------------------------------- #
# Small workloads: every row and every output against the oracle               #
# --------------------------------------------------------------------------- #

SMALL = {
    "pr1_tiny": W.pr1_tiny(),
    "compress_only_small": W.scaled(W.compress_only(), num_tokens=4999, num_blocks=400),
    "paged_decode_small": W.scaled(W.paged_decode(), batch=4, seq_len_range=(100, 600)),
    "wide_head_small": W.scaled(W.wide_head_decode(), batch=2, seq_len=700),
}
for _kb, _vb in W.LAYER_BIT_PAIRS:
    SMALL[f"mixed_k{_kb}v{_vb}_small"] = W.scaled(W.long_context_mixed(), batch=2, seq_len=333, layers=1,
                                                  layer_bits=(), k_bits=_kb, v_bits=_vb)


@pytest.mark.parametrize("name", list(SMALL))
def test_small_compress_and_decode(name):
    w = SMALL[name]
    b = W.generate(w, device="cpu")
    b = W.Batch(**{f: (getattr(b, f).to(DEV) if isinstance(getattr(b, f), torch.Tensor) else getattr(b, f))
                   for f in b.__dataclass_fields__})
    codec, ora = _codec_pair(w)
    kc, vc = _compress(codec, w, b)
    assert codec.get_status() == 0
    stats = _check_rows(ora, w, b, kc, vc)
    # whole-cache bytes: the oracle writes the same pools (same canary fill)
    geo = ora.geometry(w.page_size)
    okc = np.full(b.num_blocks * w.num_kv_heads * geo["k_page"], 0xA5, np.uint8)
    ovc = np.full(b.num_blocks * w.num_kv_heads * geo["v_page"], 0xA5, np.uint8)
    ora.compress_kv(W.as_u16(b.k), W.as_u16(b.v), b.slot_mapping.cpu().numpy(), w.page_size, b.num_blocks, okc, ovc)
    assert np.array_equal(vc.cpu().numpy(), ovc)
    if stats["code_mismatch"] == 0 and stats["norm_ulp"] == 0 and stats.get("sign_mismatch", 0) == 0 \
            and stats.get("gamma_ulp", 0) == 0:
        assert np.array_equal(kc.cpu().numpy(), okc)
    if not w.decode:
        return
    kc_np, vc_np = kc.cpu().numpy(), vc.cpu().numpy()
    out = _decode_gpu(codec, w, b, kc, vc)
    # (i) on the GPU-written cache: isolates the decode kernel
    check_decode(out, _decode_oracle(ora, w, b, kc_np, vc_np))
    # (ii) end to end: oracle's own cache
    check_decode(out, _decode_oracle(ora, w, b, okc, ovc))
    assert codec.get_status() == 0


@pytest.mark.parametrize("name", ["pr1_tiny", "mixed_k2v2_small", "mixed_k4v4_small"])
def test_tiny_magnitudes_take_the_exact_paths(name):
    """Keys below the fast path's power-of-two row scale are re-decided exactly (every
    such row, many per 128-row tile); values whose group minimum is not an fp16
    normal number are quantised by the exact value path.  Both must still match
    the oracle bit for bit."""
    w = SMALL[name]
    b = W.generate(w, device="cpu")
    T = b.k.shape[0]
    tiny = torch.zeros(T, dtype=torch.bool)
    tiny[::3] = True          # keys around 1e-36: beyond the row scale, rows redone exactly
    small = torch.zeros(T, dtype=torch.bool)
    small[1::3] = True        # values around 1e-6: fp16 subnormal zero points
    k = b.k.float()
    k[tiny] *= 1e-36
    v = b.v.float()
    v[small] *= 1e-6
    b.k, b.v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    b = W.Batch(**{f: (getattr(b, f).to(DEV) if isinstance(getattr(b, f), torch.Tensor) else getattr(b, f))
                   for f in b.__dataclass_fields__})
    codec, ora = _codec_pair(w)
    kc, vc = _compress(codec, w, b)
    assert codec.get_status() == 0
    _check_rows(ora, w, b, kc, vc)
    geo = ora.geometry(w.page_size)
    ovc = np.full(b.num_blocks * w.num_kv_heads * geo["v_page"], 0xA5, np.uint8)
    okc = np.full(b.num_blocks * w.num_kv_heads * geo["k_page"], 0xA5, np.uint8)
    ora.compress_kv(W.as_u16(b.k), W.as_u16(b.v), b.slot_mapping.cpu().numpy(), w.page_size, b.num_blocks, okc, ovc)
    assert np.array_equal(vc.cpu().numpy(), ovc)


@pytest.mark.parametrize("kb,vb,hkv", [(3, 2, 3), (4, 4, 5), (2, 3, 1)])
def test_head_counts_not_a_power_of_two(kb, vb, hkv):
    """Rows map to (token, head) by division when the head count is not a power of
    two (and by a shift when it is); tiles then start inside a token."""
    w = W.scaled(W.long_context_mixed(), batch=2, seq_len=700, layers=1, layer_bits=(), k_bits=kb, v_bits=vb,
                 num_kv_heads=hkv, num_q_heads=2 * hkv)
    b = W.generate(w, device=DEV)
    codec, ora = _codec_pair(w)
    kc, vc = _compress(codec, w, b)
    assert codec.get_status() == 0
    _check_rows(ora, w, b, kc, vc)
    out = _decode_gpu(codec, w, b, kc, vc)
    check_decode(out, _decode_oracle(ora, w, b, kc.cpu().numpy(), vc.cpu().numpy()))


def test_deferred_list_overflows_mid_kernel():
    """A third of the tokens with keys around 1e-36: ~43 rows of every 128-row tile
    take the exact path, so each CTA's 256-row deferred list fills after six tiles
    and is drained by the epilogue between tiles, the rest at the end of the
    kernel.  Sampled records (tiny and normal rows) must match the oracle."""
    w = W.scaled(W.long_context_mixed(), batch=1, seq_len=20000, layers=1, layer_bits=(), k_bits=3, v_bits=2)
    b = W.generate(w, device=DEV)
    k = b.k.float()
    k[::3] *= 1e-36
    b.k = k.to(torch.bfloat16)
    codec, ora = _codec_pair(w)
    kc, vc = _compress(codec, w, b)
    assert codec.get_status() == 0
    rng = np.random.default_rng(5)
    T = b.num_tokens
    tok = np.unique(np.concatenate([rng.integers(0, T, 1500), np.arange(0, 300), [T - 1]]))
    _check_rows(ora, w, b, kc, vc, tok)


@pytest.mark.parametrize("name", ["pr1_tiny", "wide_head_small", "mixed_k2v2_small"])
def test_dequant_matches_oracle(name):
    w = SMALL[name]
    b = W.generate(w, device="cpu")
    codec, ora = _codec_pair(w)
    k, v, sm = b.k.to(DEV), b.v.to(DEV), b.slot_mapping.to(DEV)
    kc, vc = codec.alloc_cache(b.num_blocks, w.num_kv_heads, w.page_size)
    codec.compress_kv(k, v, sm, kc, vc, w.page_size, b.num_blocks)
    slots = sm[:: max(1, len(sm) // 97)].contiguous()
    ko, vo = codec.dequant_kv(kc, vc, w.page_size, b.num_blocks, w.num_kv_heads, slots)
    torch.cuda.synchronize()
    rk, rv = ora.dequant_slots(kc.cpu().numpy(), vc.cpu().numpy(), w.page_size, w.num_kv_heads, slots.cpu().numpy())
    for got, ref in ((ko, rk), (vo, rv)):
        g = O.bf16_to_double(W.as_u16(got))
        ax = np.abs(ref)
        ulp = 2.0 ** (np.floor(np.log2(np.where(ax > 0, ax, 1.0))) - 7)
        assert np.all(np.abs(g - ref) <= ulp + 1e-5)


# --------------------------------------------------------------------------- #
# Decode edge cases                                                             #
# --------------------------------------------------------------------------- #

def _small_case(seq_lens, w=None):
    w = w or SMALL["paged_decode_small"]
    w = W.scaled(w, batch=len(seq_lens), seq_len_range=None, seq_len=max(max(seq_lens), 1))
    b = W.generate(w, device=DEV)
    b.seq_lens = torch.tensor(seq_lens, dtype=torch.int32, device=DEV)
    return w, b


def test_decode_split_counts_agree():
    w, b = _small_case([1000, 17, 640, 1])
    codec, ora = _codec_pair(w)
    kc, vc = _compress(codec, w, b)
    raw = [_decode_gpu(codec, w, b, kc, vc, splits=s) for s in (1, 2, 7, 64)]
    outs = [O.bf16_to_double(r) for r in raw]
    ax = np.abs(outs[0])
    ulp = 2.0 ** (np.floor(np.log2(np.where(ax > 0, ax, 1.0))) - 7)
    # the split count changes only the fp32 merge order and which fp16-rounded
    # probabilities meet in one accumulator: results agree to fp16 level
    for o in outs[1:]:
        assert np.all(np.abs(o - outs[0]) <= 5e-4 + ulp)
    ref = _decode_oracle(ora, w, b, kc.cpu().numpy(), vc.cpu().numpy())
    for r in raw:
        check_decode(r, ref)


def test_decode_empty_and_single_token():
    w, b = _small_case([0, 1, 5])
    codec, ora = _codec_pair(w)
    kc, vc = _compress(codec, w, b)
    out = O.bf16_to_double(_decode_gpu(codec, w, b, kc, vc))
    assert not out[0].any()
    slot = int(b.block_table[1, 0]) * w.page_size
    _, V = ora.dequant_slots(kc.cpu().numpy(), vc.cpu().numpy(), w.page_size, w.num_kv_heads, [slot])
    G = w.num_q_heads // w.num_kv_heads
    ref = np.stack([V[0, h // G] for h in range(w.num_q_heads)])
    assert np.array_equal(out[1], O.bf16_to_double(O.bf16_from_double(ref)))


@pytest.mark.parametrize("P", [16, 32])
def test_decode_round_remainders(P):
    """Each warp of a decode CTA fetches 32-token rounds w, w + 4, ... of its
    split: lengths and split counts chosen so that splits end inside a round,
    inside a page, and after fewer rounds than warps."""
    lens = [12 * P + 1, 5 * P, 31, 33, 9 * P - 1, 2 * P + 7, 3 * P]
    w, b = _small_case(lens, W.scaled(SMALL["paged_decode_small"], page_size=P))
    codec, ora = _codec_pair(w)
    kc, vc = _compress(codec, w, b)
    ref = _decode_oracle(ora, w, b, kc.cpu().numpy(), vc.cpu().numpy())
    for s in (1, 3, 5):
        check_decode(_decode_gpu(codec, w, b, kc, vc, splits=s), ref)


@pytest.mark.parametrize("name", ["mixed_k3v2_small", "mixed_k4v4_small", "wide_head_small"])
def test_strided_token_rows(name):
    """K and V whose token stride exceeds heads x head_dim (views into wider
    buffers, as in fused QKV projections) give the same records as contiguous ones."""
    w = SMALL[name]
    b = W.generate(w, device="cpu")
    T, H, d = b.k.shape
    kw = torch.zeros(T, H + 3, d, dtype=torch.bfloat16)
    vw = torch.zeros(T, H + 1, d, dtype=torch.bfloat16)
    kw[:, 1:H + 1] = b.k
    vw[:, :H] = b.v
    b = W.Batch(**{f: (getattr(b, f).to(DEV) if isinstance(getattr(b, f), torch.Tensor) else getattr(b, f))
                   for f in b.__dataclass_fields__})
    ks, vs = kw.to(DEV)[:, 1:H + 1], vw.to(DEV)[:, :H]
    assert ks.stride(0) == (H + 3) * d and vs.stride(0) == (H + 1) * d
    codec, _ = _codec_pair(w)
    kc_ref, vc_ref = _compress(codec, w, b)
    kc, vc = codec.alloc_cache(b.num_blocks, w.num_kv_heads, w.page_size, fill=0xA5)
    codec.compress_kv(ks, vs, b.slot_mapping, kc, vc, w.page_size, b.num_blocks)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    assert torch.equal(kc, kc_ref) and torch.equal(vc, vc_ref)


# compress paths: the fused tensor-core kernel (QJL keys), its keys-only form with
# the value kernel (4-bit keys), and its keys-only form twice (MSE-coded values)
COMPRESS_PATHS = [("paged_decode_small", "group"), ("mixed_k4v4_small", "group"), ("paged_decode_small", "mse")]


@pytest.mark.parametrize("name,values", COMPRESS_PATHS)
def test_bad_ids_set_status_and_write_nothing_out_of_bounds(name, values):
    w = SMALL[name]
    b = W.generate(w, device=DEV)
    codec = Codec(w.head_dim, w.k_bits, w.v_bits, w.group, w.codec_seed(), values=values)
    kpb, vpb = codec.cache_layout(w.page_size)
    guard = 4096
    kbig = torch.full((guard * 2 + b.num_blocks * w.num_kv_heads * kpb,), 0x5A, dtype=torch.uint8, device=DEV)
    vbig = torch.full((guard * 2 + b.num_blocks * w.num_kv_heads * vpb,), 0x5A, dtype=torch.uint8, device=DEV)
    kc, vc = kbig[guard:-guard], vbig[guard:-guard]
    sm = b.slot_mapping.clone()
    sm[3] = b.num_blocks * w.page_size + 5     # out of range
    sm[4] = -1                                  # skipped
    codec.compress_kv(b.k, b.v, sm, kc, vc, w.page_size, b.num_blocks)
    assert codec.get_status() & 0x1
    assert codec.get_status() == 0  # cleared by the read
    for big in (kbig, vbig):
        assert torch.all(big[:guard] == 0x5A) and torch.all(big[-guard:] == 0x5A)
    bt = b.block_table.clone()
    bt[0, 0] = b.num_blocks + 3
    out = codec.decode_attention(b.q, kc, vc, bt, b.seq_lens, w.num_kv_heads, w.page_size, b.num_blocks, b.sm_scale)
    st = codec.get_status()
    assert st & 0x2
    assert torch.isfinite(out.float()).all()
    sl = b.seq_lens.clone()
    sl[1] = bt.shape[1] * w.page_size + 100     # longer than its block table
    codec.decode_attention(b.q, kc, vc, b.block_table, sl, w.num_kv_heads, w.page_size, b.num_blocks, b.sm_scale)
    assert codec.get_status() & 0x4


def test_runs_are_deterministic_and_graph_capturable():
    w = SMALL["paged_decode_small"]
    b = W.generate(w, device=DEV)
    codec, _ = _codec_pair(w)
    kc1, vc1 = _compress(codec, w, b)
    kc2, vc2 = _compress(codec, w, b)
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    splits = codec.decode_splits(w.batch, w.num_kv_heads, b.block_table.shape[1], w.page_size)
    ws = codec.workspace(w.batch, w.num_q_heads, splits)
    out = torch.empty_like(b.q)
    ref = codec.decode_attention(b.q, kc1, vc1, b.block_table, b.seq_lens, w.num_kv_heads, w.page_size,
                                 b.num_blocks, b.sm_scale, splits=splits, workspace=ws).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        codec.decode_attention(b.q, kc1, vc1, b.block_table, b.seq_lens, w.num_kv_heads, w.page_size,
                               b.num_blocks, b.sm_scale, splits=splits, workspace=ws, out=out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    # compression captured in a graph writes the same records
    kc3, vc3 = codec.alloc_cache(b.num_blocks, w.num_kv_heads, w.page_size, fill=0xA5)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        codec.compress_kv(b.k, b.v, b.slot_mapping, kc3, vc3, w.page_size, b.num_blocks, stream=s)
    g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(kc3, kc1) and torch.equal(vc3, vc1)


# --------------------------------------------------------------------------- #
# Full-size workloads, benchmark launch configuration, sampled checks          #
# --------------------------------------------------------------------------- #

def _full_case(w, layer, n_rows=3000, n_jobs=6, seed=0):
    lw = w.for_layer(layer)
    b = W.generate(lw, layer=layer, device=DEV)
    codec, ora = _codec_pair(lw, layer)
    kc, vc = _compress(codec, lw, b, fill=0)
    assert codec.get_status() == 0
    rng = np.random.default_rng(seed)
    T = b.num_tokens
    tok = np.unique(np.concatenate([rng.integers(0, T, n_rows), [0, T - 1]]))
    _check_rows(ora, lw, b, kc, vc, tok)
    if lw.decode:
        out = _decode_gpu(codec, lw, b, kc, vc)
        jobs = [(int(rng.integers(0, lw.batch)), int(rng.integers(0, lw.num_kv_heads))) for _ in range(n_jobs)]
        jobs = sorted(set(jobs))
        ref = _decode_oracle(ora, lw, b, kc.cpu().numpy(), vc.cpu().numpy(), jobs=jobs)
        rows = _rows_of_jobs(lw, jobs)
        idx = tuple(np.array(rows).T)
        check_decode(out[idx], ref[idx])
    del kc, vc, b
    torch.cuda.empty_cache()


def test_full_compress_only():
    _full_case(W.compress_only(), 0)


def test_full_paged_decode():
    _full_case(W.paged_decode(), 0)


def test_full_wide_head_decode():
    _full_case(W.wide_head_decode(), 0)


@pytest.mark.parametrize("layer", range(8))
def test_full_long_context_mixed(layer):
    _full_case(W.long_context_mixed(), layer, n_rows=1500, n_jobs=3)


# --------------------------------------------------------------------------- #
# Barrier waits that run out                                                    #
# --------------------------------------------------------------------------- #

def test_wait_timeouts_report_and_recover():
    """With a wait limit of 0 every barrier wait tests once and gives up if its
    phase has not completed: the first page-copy wait of each decode warp and the
    first hand-off wait of each compress CTA certainly have not.  The kernels must
    set TQ_DEVERR_TIMEOUT, wind down (copies and tensor-core work in flight are
    drained with their own bound) and leave the context usable: with the default
    limit restored, both calls give the normal results again.  No wait is made to
    hang: nothing here blocks longer than the fixed drain bound."""
    from rotated_codebook_kv_gb300 import native
    w = SMALL["paged_decode_small"]
    b = W.generate(w, device=DEV)
    codec, _ = _codec_pair(w)
    kc, vc = _compress(codec, w, b)
    ref = _decode_gpu(codec, w, b, kc, vc)
    codec.set_wait_limit(0)
    out = _decode_gpu(codec, w, b, kc, vc)
    assert codec.get_status() & native.TQ_DEVERR_TIMEOUT
    assert np.all(np.isfinite(O.bf16_to_double(out)))
    kc2, vc2 = codec.alloc_cache(b.num_blocks, w.num_kv_heads, w.page_size, fill=0xA5)
    codec.compress_kv(b.k, b.v, b.slot_mapping, kc2, vc2, w.page_size, b.num_blocks)
    assert codec.get_status() & native.TQ_DEVERR_TIMEOUT
    codec.set_wait_limit(native.TQ_DEFAULT_WAIT_LIMIT)
    assert np.array_equal(_decode_gpu(codec, w, b, kc, vc), ref)
    kc3, vc3 = _compress(codec, w, b)
    assert codec.get_status() == 0
    assert torch.equal(kc3, kc) and torch.equal(vc3, vc)


@pytest.mark.parametrize("name,values", COMPRESS_PATHS[1:])
def test_compress_wait_timeouts_on_the_keys_only_paths(name, values):
    """The keys-only form of the tensor-core kernel (4-bit keys with the value
    kernel; MSE-coded values, run twice) under a wait limit of 0: its epilogue's
    first hand-off wait cannot have completed (the producers must load the tile
    first), so it reports TQ_DEVERR_TIMEOUT and winds down; with the default limit
    restored the same call writes the same bytes as before."""
    from rotated_codebook_kv_gb300 import native
    w = SMALL[name]
    b = W.generate(w, device=DEV)
    codec = Codec(w.head_dim, w.k_bits, w.v_bits, w.group, w.codec_seed(), values=values)
    kc, vc = _compress(codec, w, b)
    assert codec.get_status() == 0
    codec.set_wait_limit(0)
    kc2, vc2 = codec.alloc_cache(b.num_blocks, w.num_kv_heads, w.page_size, fill=0xA5)
    codec.compress_kv(b.k, b.v, b.slot_mapping, kc2, vc2, w.page_size, b.num_blocks)
    torch.cuda.synchronize()
    assert codec.get_status() & native.TQ_DEVERR_TIMEOUT
    codec.set_wait_limit(native.TQ_DEFAULT_WAIT_LIMIT)
    kc3, vc3 = _compress(codec, w, b)
    assert codec.get_status() == 0
    assert torch.equal(kc3, kc) and torch.equal(vc3, vc)


# --------------------------------------------------------------------------- #
# Randomized Hadamard rotation                                                  #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("d,kb,vb,g,P,G", [(128, 3, 2, 32, 16, 4), (128, 4, 4, 64, 16, 8), (256, 4, 4, 64, 32, 2),
                                           (256, 2, 3, 32, 16, 3), (256, 3, 2, 128, 32, 1)])
def test_hadamard_rotation(d, kb, vb, g, P, G):
    """The same records, decode and dequant with Pi = H D / sqrt(d): at head_dim 128
    through the tensor-core kernel (Pi as its B operand), at 256 through the
    butterfly kernel; the rotation tables equal the oracle's."""
    from rotated_codebook_kv_gb300 import native
    Hkv = 2
    w = W.Workload("hadamard", d, kb, vb, g, P, num_kv_heads=Hkv, num_q_heads=Hkv * G, batch=3,
                   seq_len_range=(200, 700), seed=d + kb)
    b = W.generate(w, device="cpu")
    b = W.Batch(**{f: (getattr(b, f).to(DEV) if isinstance(getattr(b, f), torch.Tensor) else getattr(b, f))
                   for f in b.__dataclass_fields__})
    codec = Codec(d, kb, vb, g, w.codec_seed(), rotation=native.TQ_ROTATION_HADAMARD)
    ora = O.Oracle(d, kb, vb, g, w.codec_seed(), rotation=O.Oracle.ROTATION_HADAMARD)
    lib, ref = codec.export_params(), ora.params()
    assert np.all(np.abs(lib["Pi"].astype(np.float64) - ref["Pi"]) <= np.abs(ref["Pi"]) * 2.0 ** -24)
    kc, vc = _compress(codec, w, b)
    assert codec.get_status() == 0
    _check_rows(ora, w, b, kc, vc)
    kc_np, vc_np = kc.cpu().numpy(), vc.cpu().numpy()
    check_decode(_decode_gpu(codec, w, b, kc, vc), _decode_oracle(ora, w, b, kc_np, vc_np))
    slots = b.slot_mapping[::7].contiguous()
    ko, vo = codec.dequant_kv(kc, vc, P, b.num_blocks, Hkv, slots)
    torch.cuda.synchronize()
    rk, _ = ora.dequant_slots(kc_np, vc_np, P, Hkv, slots.cpu().numpy())
    gk = O.bf16_to_double(W.as_u16(ko))
    ax = np.abs(rk)
    ulp = 2.0 ** (np.floor(np.log2(np.where(ax > 0, ax, 1.0))) - 7)
    assert np.all(np.abs(gk - rk) <= ulp + 1e-5)


@pytest.mark.parametrize("vb,g", [(4, 64), (2, 32), (3, 128)])
def test_hadamard_streaming_kernel_special_rows(vb, g):
    """head_dim 256, 4-bit keys, Hadamard rotation (the streaming kernel): zero keys,
    keys around 1e-36 and around 1e30 (redone in double), constant and zero value
    groups, and values whose minimum is an fp16 subnormal match the oracle."""
    from rotated_codebook_kv_gb300 import native
    d, kb, P, Hkv = 256, 4, 32, 2
    w = W.Workload("hadamard_stream", d, kb, vb, g, P, num_kv_heads=Hkv, num_q_heads=Hkv * 2, batch=2,
                   seq_len_range=(300, 500), seed=77 + vb)
    b = W.generate(w, device="cpu")
    k, v = b.k.float(), b.v.float()
    k[3] = 0.0
    k[10::17] *= 1e-36
    k[11::29] *= 1e30
    v[5, :, :g] = 2.5
    v[6] = 0.0
    v[12::13] *= 1e-6
    b.k, b.v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    b = W.Batch(**{f: (getattr(b, f).to(DEV) if isinstance(getattr(b, f), torch.Tensor) else getattr(b, f))
                   for f in b.__dataclass_fields__})
    codec = Codec(d, kb, vb, g, w.codec_seed(), rotation=native.TQ_ROTATION_HADAMARD)
    ora = O.Oracle(d, kb, vb, g, w.codec_seed(), rotation=O.Oracle.ROTATION_HADAMARD)
    kc, vc = _compress(codec, w, b)
    assert codec.get_status() == 0
    _check_rows(ora, w, b, kc, vc)
    geo = ora.geometry(P)
    okc = np.full(b.num_blocks * Hkv * geo["k_page"], 0xA5, np.uint8)
    ovc = np.full(b.num_blocks * Hkv * geo["v_page"], 0xA5, np.uint8)
    ora.compress_kv(W.as_u16(b.k), W.as_u16(b.v), b.slot_mapping.cpu().numpy(), P, b.num_blocks, okc, ovc)
    assert np.array_equal(vc.cpu().numpy(), ovc)


# --------------------------------------------------------------------------- #
# Sizes at the edges of what the calls accept                                   #
# --------------------------------------------------------------------------- #

def test_size_edges():
    """Empty calls launch nothing and touch nothing; the largest accepted split count
    (1024, far more splits than pages) decodes correctly; 65535 sequences (the
    largest batch) of length 0 and 1 decode to zeros and to their single value;
    one past the largest batch and split count is refused on the host."""
    from rotated_codebook_kv_gb300 import native
    w = W.scaled(SMALL["paged_decode_small"], batch=3, seq_len_range=(50, 120))
    b = W.generate(w, device=DEV)
    codec, ora = _codec_pair(w)
    kc, vc = _compress(codec, w, b, fill=0x3C)
    before = (kc.clone(), vc.clone())
    codec.compress_kv(b.k[:0], b.v[:0], b.slot_mapping[:0], kc, vc, w.page_size, b.num_blocks)  # T = 0
    torch.cuda.synchronize()
    assert torch.equal(kc, before[0]) and torch.equal(vc, before[1])
    ref = _decode_oracle(ora, w, b, kc.cpu().numpy(), vc.cpu().numpy())
    check_decode(_decode_gpu(codec, w, b, kc, vc, splits=1024), ref)
    assert codec.get_status() == 0
    # the largest batch: 65535 sequences, alternately empty and of one token (the first slot of a page)
    Bmax = 65535
    q = torch.randn(Bmax, w.num_q_heads, w.head_dim, device=DEV).to(torch.bfloat16)
    bt = torch.zeros(Bmax, 1, dtype=torch.int32, device=DEV)
    bt[:, 0] = b.block_table[0, 0]
    sl = (torch.arange(Bmax, device=DEV, dtype=torch.int32) % 2)
    out = codec.decode_attention(q, kc, vc, bt, sl, w.num_kv_heads, w.page_size, b.num_blocks, b.sm_scale)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    o = O.bf16_to_double(W.as_u16(out))
    assert not o[0::2].any()
    _, V = ora.dequant_slots(kc.cpu().numpy(), vc.cpu().numpy(), w.page_size, w.num_kv_heads,
                             [int(b.block_table[0, 0]) * w.page_size])
    G = w.num_q_heads // w.num_kv_heads
    want = O.bf16_to_double(O.bf16_from_double(np.stack([V[0, h // G] for h in range(w.num_q_heads)])))
    assert np.array_equal(o[1], want) and np.array_equal(o[-2], want)
    ws = codec.workspace(1, w.num_q_heads, 1)
    with pytest.raises(native.TQError):  # one sequence too many
        native.tq_decode_attention(codec.handle, q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
                                   sl.data_ptr(), Bmax + 1, w.num_q_heads, w.num_kv_heads, w.page_size, 1,
                                   b.num_blocks, b.sm_scale, 1, ws.data_ptr(), ws.numel(), out.data_ptr(), 0)
    with pytest.raises(native.TQError):  # one split too many
        native.tq_decode_attention(codec.handle, q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
                                   sl.data_ptr(), 1, w.num_q_heads, w.num_kv_heads, w.page_size, 1,
                                   b.num_blocks, b.sm_scale, 1025, ws.data_ptr(), ws.numel(), out.data_ptr(), 0)


# --------------------------------------------------------------------------- #
# Query rotation on the tensor cores (many query rows)                         #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("d,kb,vb,G", [(128, 3, 2, 8), (128, 4, 4, 4), (256, 2, 3, 4), (256, 4, 2, 8)])
def test_many_query_rows_use_the_tensor_core_rotation(d, kb, vb, G):
    """A call with at least 2,048 query rows rotates the queries with mma.sync (Pi 2^10
    and M = S Pi as fp16 high/low fragments) instead of the fp32 kernel; decode through
    it (with and without QJL, both head dims, one split and several) still matches the
    oracle element by element, and the rotation equals the fp32 path's to 2^-16 of its
    largest element (both are ~2^-22-accurate products; a wrong matrix errs by O(1))."""
    Hkv = 4
    B = 2048 // (Hkv * G) + 3
    w = W.Workload("many_rows", d, kb, vb, 32, 16, num_kv_heads=Hkv, num_q_heads=Hkv * G, batch=B,
                   seq_len_range=(20, 90), seed=d + kb + G)
    b = W.generate(w, device="cpu")
    b = W.Batch(**{f: (getattr(b, f).to(DEV) if isinstance(getattr(b, f), torch.Tensor) else getattr(b, f))
                   for f in b.__dataclass_fields__})
    codec = Codec(d, kb, vb, 32, w.codec_seed())
    ora = O.Oracle(d, kb, vb, 32, w.codec_seed())
    kc, vc = _compress(codec, w, b)
    kc_np, vc_np = kc.cpu().numpy(), vc.cpu().numpy()
    ref = _decode_oracle(ora, w, b, kc_np, vc_np)
    for splits in (1, 3):
        check_decode(_decode_gpu(codec, w, b, kc, vc, splits=splits), ref)
    assert codec.get_status() == 0
    # the rotated queries themselves: fp32 workspace rows after a call with many rows
    # against a call with few (the fp32 kernel), sequence by sequence
    rows = B * w.num_q_heads
    ws = codec.workspace(B, w.num_q_heads, 1, device=DEV)
    codec.decode_attention(b.q, kc, vc, b.block_table, b.seq_lens, Hkv, 16, b.num_blocks, b.sm_scale, splits=1,
                           workspace=ws)
    torch.cuda.synchronize()
    wsf = ws.view(torch.float32)
    al = lambda x: (x + 63) // 64 * 64  # 256-byte pieces, in floats
    qrot_many = wsf[al(rows * d): al(rows * d) + rows * d].clone()
    ws1 = codec.workspace(1, w.num_q_heads, 1, device=DEV)
    qrot_few = torch.empty_like(qrot_many)
    for s in range(B):
        codec.decode_attention(b.q[s:s + 1].contiguous(), kc, vc, b.block_table[s:s + 1].contiguous(),
                               b.seq_lens[s:s + 1].contiguous(), Hkv, 16, b.num_blocks, b.sm_scale, splits=1,
                               workspace=ws1)
        r1 = w.num_q_heads
        qrot_few[s * r1 * d:(s + 1) * r1 * d] = ws1.view(torch.float32)[al(r1 * d): al(r1 * d) + r1 * d]
    torch.cuda.synchronize()
    scale = qrot_few.abs().max()
    assert float((qrot_many - qrot_few).abs().max()) <= float(scale) * 2.0 ** -16


@pytest.mark.parametrize("d,kb,vb,g,values", [(128, 3, 2, 32, "group"), (128, 4, 4, 64, "group"),
                                              (256, 2, 3, 32, "group"), (128, 2, 3, 32, "mse"),
                                              (256, 4, 2, 64, "mse")])
def test_dequant_many_slots_on_the_tensor_cores(d, kb, vb, g, values):
    """tq_dequant_kv over thousands of (slot, kv head) rows runs on mma.sync (Pi^T and
    S^T as fp16 high/low fragment images); every reconstructed element is within one
    bf16 ulp of the oracle's double-precision dequantisation, or 2^-20 of its row's
    norm for elements near zero (the products carry ~22 bits: measured worst 1.4e-7 of
    the norm), skipped slots (-1) are left untouched, and a second call with a few
    slots (the CUDA-core kernel) agrees to the same bound."""
    Hkv = 2
    w = W.Workload("dq_many", d, kb, vb, g, 16, num_kv_heads=Hkv, num_q_heads=Hkv, batch=8,
                   seq_len_range=(250, 450), seed=3 * d + kb + vb)
    b = W.generate(w, device="cpu")
    b = W.Batch(**{f: (getattr(b, f).to(DEV) if isinstance(getattr(b, f), torch.Tensor) else getattr(b, f))
                   for f in b.__dataclass_fields__})
    codec = Codec(d, kb, vb, g, w.codec_seed(), values=values)
    ora = O.Oracle(d, kb, vb, g, w.codec_seed(), values=values)
    kc, vc = codec.alloc_cache(b.num_blocks, Hkv, 16, fill=0xA5)
    codec.compress_kv(b.k, b.v, b.slot_mapping, kc, vc, 16, b.num_blocks)
    slots = b.slot_mapping.clone()
    slots[5] = -1
    assert slots.numel() * Hkv >= 2048
    ko = torch.full((slots.numel(), Hkv, d), 0x7FC1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    vo = torch.full_like(ko, 0)
    vo.view(torch.int16).fill_(0x7FC1)
    codec.dequant_kv(kc, vc, 16, b.num_blocks, Hkv, slots, k_out=ko, v_out=vo)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    rk, rv = ora.dequant_slots(kc.cpu().numpy(), vc.cpu().numpy(), 16, Hkv, slots.cpu().numpy())
    gk, gv = O.bf16_to_double(W.as_u16(ko)), O.bf16_to_double(W.as_u16(vo))
    keep = np.ones(slots.numel(), dtype=bool)
    keep[5] = False
    def bound(ref):
        ax = np.abs(ref)
        ulp = 2.0 ** (np.floor(np.log2(np.where(ax > 0, ax, 1.0))) - 7)
        return ulp + 2.0 ** -20 * np.linalg.norm(ref, axis=-1, keepdims=True)
    for gg, rr_ in ((gk, rk), (gv, rv)):
        assert np.all(np.abs(gg[keep] - rr_[keep]) <= bound(rr_[keep]))
    assert np.all(W.as_u16(ko)[5] == 0x7FC1) and np.all(W.as_u16(vo)[5] == 0x7FC1)
    few = slots[:40].contiguous()
    kf, vf = codec.dequant_kv(kc, vc, 16, b.num_blocks, Hkv, few)
    torch.cuda.synchronize()
    m = np.ones(40, dtype=bool)
    m[5] = False
    for a_, r_ in ((kf, rk[:40]), (vf, rv[:40])):
        assert np.all(np.abs(O.bf16_to_double(W.as_u16(a_))[m] - r_[m]) <= bound(r_[m]))
