"""Pins of the oracle's codec (key/value records, page layout, dequant, decode).

What fixes each expected value:
* key MSE: the Lloyd-Max distortion of N(0,1) at b bits (J. Max 1960, Table I),
  since rotated unit-vector coordinates scaled by sqrt(d) are ~N(0,1)
  (brightcoding blog, "What is TurboQuant-GPU?": rotation makes coordinates
  approximately Gaussian, where Lloyd-Max is optimal);
* QJL: the 1-bit sign sketch of the residual gives an unbiased inner-product
  estimate (0xsero/turboquant, "Operational Constraints": near-unbiased
  approximate inner products) -- checked by Monte Carlo over independent S;
* values: per-group min/max affine quantisation (0xsero/turboquant "Value
  Compression"; tiny-turboquant "Measured quality": one scale/zero pair per
  group) -- numpy's own float16 rounding and exact rational arithmetic;
* compression ratios: the figures printed on the brightcoding blog, rebuilt
  from the oracle's record sizes (tests/golden/compression_ratios.json);
* decode: dense softmax attention over the dequantised cache (numpy), the
  rotated-space identity <Pi q, Pi k> = <q, k>, and closed-form special cases.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MAX_MSE = {2: 0.1175, 3: 0.03454, 4: 0.009497}


def _bf16(x):
    """float64 array -> bf16 bit patterns (round to nearest even via float32 of exact bf16 grid)."""
    return O.bf16_from_double(np.asarray(x, dtype=np.float64))


# --------------------------------------------------------------------------- #
# Keys                                                                           #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("bits", [2, 3, 4])
def test_key_codebook_distortion_matches_lloyd_max(bits):
    d = 128
    ora = O.Oracle(d, bits, 4, 32, seed=1)
    rng = np.random.default_rng(bits)
    k = _bf16(rng.standard_normal((4000, d)))
    rec = ora.compress_rows(k=k)
    c = ora.params()["centroids"]
    codes = np.stack([O.unpack(r, d, bits) for r in rec["k_code"]])
    mse = np.mean((rec["z"] - c[codes]) ** 2)
    assert abs(mse - MAX_MSE[bits]) < 0.05 * MAX_MSE[bits]
    # the stored norm is the bf16 rounding of ||k||
    kd = O.bf16_to_double(k)
    assert np.array_equal(rec["k_norm"], _bf16(np.linalg.norm(kd, axis=1)))


def test_key_zero_vector_gives_zero_record():
    ora = O.Oracle(128, 3, 4, 32, seed=0)
    rec = ora.compress_rows(k=np.zeros((2, 128), np.uint16))
    for f in ("k_code", "k_sign", "k_norm", "k_gamma"):
        assert not rec[f].any()


def test_qjl_gamma_is_residual_norm():
    d = 128
    ora = O.Oracle(d, 2, 4, 32, seed=2)
    rng = np.random.default_rng(5)
    k = _bf16(rng.standard_normal((64, d)))
    rec = ora.compress_rows(k=k)
    c = ora.params()["centroids"]
    codes = np.stack([O.unpack(r, d, 2) for r in rec["k_code"]])
    r = (rec["z"] - c[codes]) / math.sqrt(d)
    assert np.allclose(rec["gamma"], np.linalg.norm(r, axis=1), rtol=1e-12)
    assert np.array_equal(rec["k_gamma"], _bf16(rec["gamma"]))


@pytest.mark.parametrize("bits", [2, 3])
def test_qjl_estimator_unbiased_monte_carlo(bits):
    """Fixed Pi, q, k; independent S: mean of <q, K~> is <q, k> (bias <= 2^-8 rel)."""
    d, P, n_mc = 32, 16, 4000
    rng = np.random.default_rng(100 + bits)
    k_d = O.bf16_to_double(_bf16(rng.standard_normal(d)))
    q = k_d + 0.5 * rng.standard_normal(d)  # aligned with k so the residual term matters
    truth = float(q @ k_d)
    kk = _bf16(k_d).reshape(1, 1, d)
    vv = np.zeros((1, 1, d), np.uint16)
    slot = np.array([0], np.int64)
    est = np.empty(n_mc)
    mse_only = None
    for s in range(n_mc):
        ora = O.Oracle(d, bits, 4, 32, seed=0, qjl_seed=1000 + s)
        kc, vc = ora.compress_kv(kk, vv, slot, P, 1)
        kt, _ = ora.dequant_slots(kc, vc, P, 1, slot)
        est[s] = q @ kt[0, 0]
        if mse_only is None:  # codebook-only reconstruction n16 * Pi^T c[code]/sqrt(d)
            prm = ora.params()
            rec = ora.compress_rows(k=kk[0])
            codes = O.unpack(rec["k_code"][0], d, bits)
            n16 = O.bf16_to_double(rec["k_norm"][0])
            mse_only = float(q @ (n16 * prm["Pi"].T @ (prm["centroids"][codes] / math.sqrt(d))))
    se = est.std(ddof=1) / math.sqrt(n_mc)
    assert abs(est.mean() - truth) < 4 * se + 2.0 ** -8 * abs(truth)
    # the residual correction is what removes the bias: without it the estimate is off
    assert abs(mse_only - truth) > 10 * se


# --------------------------------------------------------------------------- #
# Values                                                                         #
# --------------------------------------------------------------------------- #

def _groups(rng, n, g):
    x = rng.standard_normal((n, g)) * np.exp(rng.standard_normal((n, 1)))
    x[0] = 1.25                     # constant group
    x[1] = 0.0                      # all zeros
    x[2, : g // 2] = -3.0           # two-valued group
    x[2, g // 2:] = 5.5
    return _bf16(x)


@pytest.mark.parametrize("vbits", [2, 3, 4])
@pytest.mark.parametrize("g", [32, 64, 128])
def test_value_group_quantisation_exact(vbits, g):
    d = 128
    ora = O.Oracle(d, 4, vbits, g, seed=0)
    rng = np.random.default_rng(vbits * 1000 + g)
    v = _groups(rng, 3 * (d // g) * 20, g).reshape(-1, d)
    rec = ora.compress_rows(v=v)
    L = (1 << vbits) - 1
    xs = O.bf16_to_double(v).reshape(len(v), d // g, g)
    codes = np.stack([O.unpack(r, d, vbits) for r in rec["v_code"]]).reshape(len(v), d // g, g)
    meta = rec["v_meta"].reshape(len(v), d // g, 2)
    mn, mx = xs.min(axis=2), xs.max(axis=2)
    # scale / zero: fp16 round-to-nearest-even of (max-min)/L and of min (numpy's rounding)
    assert np.array_equal(meta[..., 0], ((mx - mn) / L).astype(np.float16).view(np.uint16))
    assert np.array_equal(meta[..., 1], mn.astype(np.float16).view(np.uint16))
    s = meta[..., 0].view(np.float16).astype(np.float64)
    z = meta[..., 1].view(np.float16).astype(np.float64)
    assert codes.max() <= L
    # exact round-half-up of (x - z)/s, checked in rational arithmetic on a sample
    for i in range(0, xs.shape[0], 7):
        for gi in range(xs.shape[1]):
            S, Z = Fraction(s[i, gi]), Fraction(z[i, gi])
            for j in range(0, g, 5):
                X = Fraction(xs[i, gi, j])
                want = 0 if S == 0 else min(max(math.floor((X - Z) / S + Fraction(1, 2)), 0), L)
                assert codes[i, gi, j] == want
    # reconstruction within half a step inside the representable range
    rec_x = codes * s[..., None] + z[..., None]
    inside = (xs >= z[..., None] - s[..., None] / 2) & (xs <= z[..., None] + (L + 0.5) * s[..., None])
    assert np.all(np.abs(rec_x - xs)[inside] <= s[..., None].repeat(g, 2)[inside] / 2 + 1e-12)
    # a constant group reconstructs exactly
    const = (mx == mn)
    assert np.all(np.abs(rec_x - xs)[np.repeat(const[..., None], g, 2)] == 0)


# --------------------------------------------------------------------------- #
# Page layout                                                                    #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("kb,vb,g,d,P", [(3, 4, 32, 128, 16), (4, 4, 64, 256, 32), (2, 2, 32, 128, 16)])
def test_page_layout_offsets(kb, vb, g, d, P):
    ora = O.Oracle(d, kb, vb, g, seed=3)
    geo = ora.geometry(P)
    qjl = kb <= 3
    assert geo["k_page"] == P * (d * kb // 8 + (d // 8 + 2 if qjl else 0) + 2)
    assert geo["v_page"] == P * (d * vb // 8 + 4 * d // g)
    for f in ("k_code", "k_sign", "v_code", "v_meta"):
        assert (P * geo[f]) % 16 == 0  # every sub-array stays 16-byte aligned
    Hkv, nb, T = 2, 3, 5
    rng = np.random.default_rng(9)
    k = _bf16(rng.standard_normal((T, Hkv, d)))
    v = _bf16(rng.standard_normal((T, Hkv, d)))
    slots = np.array([P + 3, 2 * P + P - 1, -1, 0, 5], np.int64)
    kc, vc = ora.compress_kv(k, v, slots, P, nb)
    rec = ora.compress_rows(k=k.reshape(-1, d), v=v.reshape(-1, d))
    kc2 = np.zeros_like(kc)
    vc2 = np.zeros_like(vc)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(int(s), P)
        for h in range(Hkv):
            i = t * Hkv + h
            kr = (blk * Hkv + h) * geo["k_page"]
            vr = (blk * Hkv + h) * geo["v_page"]
            kc2[kr + off * geo["k_code"]: kr + (off + 1) * geo["k_code"]] = rec["k_code"][i]
            base = kr + P * geo["k_code"]
            if qjl:
                kc2[base + off * geo["k_sign"]: base + (off + 1) * geo["k_sign"]] = rec["k_sign"][i]
            base += P * geo["k_sign"]
            kc2[base + 2 * off: base + 2 * off + 2] = np.array([rec["k_norm"][i]], np.uint16).view(np.uint8)
            if qjl:
                base += 2 * P
                kc2[base + 2 * off: base + 2 * off + 2] = np.array([rec["k_gamma"][i]], np.uint16).view(np.uint8)
            vc2[vr + off * geo["v_code"]: vr + (off + 1) * geo["v_code"]] = rec["v_code"][i]
            base = vr + P * geo["v_code"]
            vc2[base + off * geo["v_meta"]: base + (off + 1) * geo["v_meta"]] = rec["v_meta"][i].view(np.uint8)
    assert np.array_equal(kc, kc2)
    assert np.array_equal(vc, vc2)


def test_compression_ratios_from_record_sizes():
    gold = json.load(open(os.path.join(GOLDEN, "compression_ratios.json")))
    d = 128
    fp16_bytes = 2 * 2 * d  # one fp16 key plus one fp16 value
    # 2-bit key codebook + QJL: key record bytes from the oracle's geometry
    k_rec = O.Oracle(d, 2, 3, 32, seed=0).geometry(16)["k_page"] // 16
    assert k_rec == 32 + 16 + 2 + 2
    # 3-bit MSE value: 3-bit codes plus one 16-bit norm, from the MSE-value record geometry
    v_rec = O.Oracle(d, 4, 3, 128, seed=0, values="mse").geometry(16)["v_page"] // 16
    assert v_rec == 48 + 2
    ratio = fp16_bytes / (k_rec + v_rec)
    assert round(ratio, 2) == gold["turboquant_2bit_k_qjl_3bit_v_vs_fp16"]["value"]
    assert round(16 / (4 + 8 / 32), 2) == gold["mxfp4_vs_fp16"]["value"]
    assert round(16 / (4 + 8 / 16), 2) == gold["nvfp4_vs_fp16"]["value"]


# --------------------------------------------------------------------------- #
# Decode                                                                         #
# --------------------------------------------------------------------------- #

def _tiny_case(d=128, kb=3, vb=4, g=32, P=16, B=3, Hkv=2, G=2, lens=(37, 16, 1), seed=4):
    ora = O.Oracle(d, kb, vb, g, seed=seed)
    rng = np.random.default_rng(seed)
    lens = np.array(lens, np.int32)
    npg = (lens + P - 1) // P
    nb = int(npg.sum()) + 2
    perm = rng.permutation(nb).astype(np.int32)
    maxb = int(npg.max())
    bt = np.full((B, maxb), -1, np.int32)
    st = 0
    for b in range(B):
        bt[b, : npg[b]] = perm[st: st + npg[b]]
        st += npg[b]
    T = int(lens.sum())
    k = _bf16(rng.standard_normal((T, Hkv, d)) * 1.5)
    v = _bf16(rng.standard_normal((T, Hkv, d)))
    slots = np.concatenate([bt[b, np.arange(lens[b]) // P].astype(np.int64) * P + np.arange(lens[b]) % P
                            for b in range(B)])
    kc, vc = ora.compress_kv(k, v, slots, P, nb)
    q = _bf16(rng.standard_normal((B, Hkv * G, d)))
    return ora, dict(q=q, kc=kc, vc=vc, bt=bt, lens=lens, P=P, Hkv=Hkv, slots=slots, d=d)


def _numpy_attention(ora, c, sm_scale):
    """Dense softmax attention over the oracle's dequantised K~, V~ (numpy)."""
    q = O.bf16_to_double(c["q"])
    B, Hq, d = q.shape
    G = Hq // c["Hkv"]
    out = np.zeros((B, Hq, d))
    for b in range(B):
        L = int(c["lens"][b])
        if L == 0:
            continue
        pos = np.arange(L)
        slots = c["bt"][b, pos // c["P"]].astype(np.int64) * c["P"] + pos % c["P"]
        K, V = ora.dequant_slots(c["kc"], c["vc"], c["P"], c["Hkv"], slots)
        for h in range(Hq):
            s = sm_scale * K[:, h // G] @ q[b, h]
            p = np.exp(s - s.max())
            out[b, h] = (p / p.sum()) @ V[:, h // G]
    return out


@pytest.mark.parametrize("kw", [dict(), dict(d=256, kb=4, vb=4, g=64, P=32, lens=(70, 33, 2)),
                                dict(kb=2, vb=2, g=32, G=4, lens=(5, 64, 17))])
def test_decode_matches_dense_attention(kw):
    ora, c = _tiny_case(**kw)
    sm = c["d"] ** -0.5
    ref = _numpy_attention(ora, c, sm)
    for mode in (0, 1):
        out = ora.decode(c["q"], c["kc"], c["vc"], c["bt"], c["lens"], c["Hkv"], c["P"], sm, mode=mode)
        assert np.abs(out - ref).max() < 1e-10 * max(1.0, np.abs(ref).max())


def test_decode_special_cases():
    ora, c = _tiny_case(lens=(1, 0, 16))
    sm = c["d"] ** -0.5
    out = ora.decode(c["q"], c["kc"], c["vc"], c["bt"], c["lens"], c["Hkv"], c["P"], sm)
    # seq_len 1: the output is the single dequantised value
    _, V = ora.dequant_slots(c["kc"], c["vc"], c["P"], c["Hkv"], [int(c["bt"][0, 0]) * c["P"]])
    for h in range(4):
        assert np.array_equal(out[0, h], V[0, h // 2])
    # seq_len 0: zeros
    assert not out[1].any()
    # zero query: uniform weights, the mean of the dequantised values
    q0 = c["q"].copy()
    q0[2] = 0
    out0 = ora.decode(q0, c["kc"], c["vc"], c["bt"], c["lens"], c["Hkv"], c["P"], sm)
    slots = c["bt"][2, 0].astype(np.int64) * c["P"] + np.arange(16)
    _, V = ora.dequant_slots(c["kc"], c["vc"], c["P"], c["Hkv"], slots)
    for h in range(4):
        assert np.allclose(out0[2, h], V[:, h // 2].mean(axis=0), atol=1e-12)


def test_decode_identical_keys_average_values():
    d, P, Hkv = 128, 16, 1
    ora = O.Oracle(d, 3, 4, 32, seed=8)
    rng = np.random.default_rng(8)
    key = _bf16(rng.standard_normal(d))
    k = np.tile(key, (20, 1)).reshape(20, 1, d)
    v = _bf16(rng.standard_normal((20, 1, d)))
    bt = np.array([[1, 0]], np.int32)
    slots = np.concatenate([np.arange(16) + 16, np.arange(4)]).astype(np.int64)
    kc, vc = ora.compress_kv(k, v, slots, P, 2)
    q = _bf16(rng.standard_normal((1, 2, d)) * 3)
    out = ora.decode(q, kc, vc, bt, np.array([20], np.int32), Hkv, P, d ** -0.5)
    _, V = ora.dequant_slots(kc, vc, P, Hkv, slots)
    assert np.allclose(out[0, 0], V[:, 0].mean(axis=0), atol=1e-12)
    assert np.allclose(out[0, 1], V[:, 0].mean(axis=0), atol=1e-12)


# --------------------------------------------------------------------------- #
# Reading records back: dequant_slots and the QJL half for given codes          #
# --------------------------------------------------------------------------- #

def _paged_rows(d, kb, vb, g, P, T=40, Hkv=3, seed=11):
    """Random keys and values (with constant and all-zero value groups) written to
    shuffled slots of a small paged pool by the oracle."""
    ora = O.Oracle(d, kb, vb, g, seed=seed)
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((T, Hkv, d)) * np.exp(rng.standard_normal((T, Hkv, 1)))
    v = rng.standard_normal((T, Hkv, d)) * np.exp(rng.standard_normal((T, Hkv, 1)))
    v[0, 0, :g] = 0.75          # a constant group
    v[1, 1, g:2 * g if 2 * g <= d else d] = 0.0  # an all-zero group (or the whole row at g = d)
    nb = (T + P - 1) // P + 2
    slots = rng.permutation(nb * P)[:T].astype(np.int64)
    kk, vv = _bf16(k), _bf16(v)
    kc, vc = ora.compress_kv(kk, vv, slots, P, nb)
    return ora, kk, vv, slots, kc, vc


@pytest.mark.parametrize("d,kb,vb,g,P", [(128, 3, 4, 32, 16), (128, 2, 2, 64, 16), (128, 4, 3, 128, 32),
                                         (256, 4, 4, 64, 32)])
def test_dequant_values_reconstruct_the_inputs(d, kb, vb, g, P):
    """V~ read back by dequant_slots: within half a quantisation step of the bf16
    input inside the group's range, exact for constant groups, and equal to
    code * scale + zero with every field decoded by numpy from the raw bytes
    (the record reader in tests/parity.py), so a slip in the group index or a
    swap of scale and zero in the read-back fails."""
    from parity import read_records
    ora, kk, vv, slots, kc, vc = _paged_rows(d, kb, vb, g, P)
    T, Hkv, _ = vv.shape
    _, V = ora.dequant_slots(kc, vc, P, Hkv, slots)
    geo = ora.geometry(P)
    rec = read_records(kc, vc, geo, d, kb, vb, g, P, Hkv, slots)
    s = rec["v_meta"][..., 0].view(np.float16).astype(np.float64)   # [T, Hkv, d/g]
    z = rec["v_meta"][..., 1].view(np.float16).astype(np.float64)
    code = rec["v_code"].astype(np.float64)                          # [T, Hkv, d]
    s_e, z_e = np.repeat(s, g, axis=-1), np.repeat(z, g, axis=-1)
    assert np.array_equal(V, code * s_e + z_e)
    x = O.bf16_to_double(vv)
    xg = x.reshape(T, Hkv, d // g, g)
    mn, mx = xg.min(-1), xg.max(-1)
    L = (1 << vb) - 1
    # half a step inside [mn, mx], plus what the fp16 roundings of zero and scale move the grid
    slack = np.abs(mn - z) + L * np.abs(s - (mx - mn) / L)
    err = np.abs(V - x).reshape(T, Hkv, d // g, g)
    assert np.all(err <= (s / 2 + slack + 1e-12)[..., None])
    const = (mx == mn)
    assert const.any()
    assert np.all(err[const] == 0.0)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_dequant_keys_rotate_back_to_the_codebook(bits):
    """K~ read back by dequant_slots, rotated by Pi (pinned orthogonal) and scaled
    by sqrt(d) / n16, gives back the centroids of the stored codes (decoded by
    numpy from the raw bytes) exactly when there is no QJL term; with QJL the
    difference is the sign-sketch correction, whose size follows from gamma and
    the Gaussian S.  Without QJL the distance to the input key is the Lloyd-Max
    distortion of the codebook (J. Max 1960)."""
    from parity import read_records
    d, P = 128, 16
    ora, kk, vv, slots, kc, vc = _paged_rows(d, bits, 4, 32, P, T=300, Hkv=2, seed=20 + bits)
    T, Hkv, _ = kk.shape
    K, _ = ora.dequant_slots(kc, vc, P, Hkv, slots)
    prm = ora.params()
    rec = read_records(kc, vc, ora.geometry(P), d, bits, 4, 32, P, Hkv, slots)
    n16 = O.bf16_to_double(rec["k_norm"])                            # [T, Hkv]
    u = np.einsum("ij,thj->thi", prm["Pi"], K) * math.sqrt(d) / n16[..., None]
    cz = prm["centroids"][rec["k_code"]]
    if bits == 4:
        assert np.abs(u - cz).max() < 1e-10
    else:
        # the QJL term sqrt(pi/2)/d * gamma * S^T(2 sigma - 1), in z units, has norm
        # about sqrt(pi/2) gamma sqrt(d) ||S^T(2 sigma - 1)|| / d ~ sqrt(pi/2) * gamma * sqrt(d)
        gam = O.bf16_to_double(rec["k_gamma"])
        corr = np.linalg.norm(u - cz, axis=-1)
        ratio = corr / (gam * math.sqrt(d) * math.sqrt(math.pi / 2))
        assert 0.7 < ratio.mean() < 1.4
    k = O.bf16_to_double(kk)
    kn = np.linalg.norm(k, axis=-1)
    rel = np.sum((K - k) ** 2, axis=-1) / kn ** 2   # = ||z - c||^2 / d: the per-coordinate MSE in z units
    if bits == 4:
        assert abs(rel.mean() - MAX_MSE[bits]) < 0.08 * MAX_MSE[bits]


@pytest.mark.parametrize("bits", [2, 3])
def test_qjl_given_codes_reproduces_the_compressor(bits):
    """The QJL half for given codes, fed the compressor's own codes, gives the
    compressor's signs, gamma and projections bit for bit; fed a code moved by one
    level on one coordinate, gamma changes exactly as the residual definition says
    (r_j = z_j / sqrt(d) - c[code_j] / sqrt(d))."""
    d = 128
    ora = O.Oracle(d, bits, 4, 32, seed=31)
    rng = np.random.default_rng(31 + bits)
    k = _bf16(rng.standard_normal((50, d)) * 2.0)
    rec = ora.compress_rows(k=k)
    codes = np.stack([O.unpack(r, d, bits) for r in rec["k_code"]])
    alt = ora.key_qjl_given_codes(k, codes)
    assert np.array_equal(alt["k_sign"], rec["k_sign"])
    assert np.array_equal(alt["k_gamma"], rec["k_gamma"])
    assert np.array_equal(alt["gamma"], rec["gamma"])
    assert np.array_equal(alt["pg"], rec["pg"])
    c = ora.params()["centroids"]
    L = 1 << bits
    moved = codes.copy()
    j = 17
    moved[:, j] = np.where(moved[:, j] + 1 < L, moved[:, j] + 1, moved[:, j] - 1)
    alt2 = ora.key_qjl_given_codes(k, moved)
    r_old = (rec["z"][:, j] - c[codes[:, j]]) / math.sqrt(d)
    r_new = (rec["z"][:, j] - c[moved[:, j]]) / math.sqrt(d)
    want = np.sqrt(rec["gamma"] ** 2 - r_old ** 2 + r_new ** 2)
    assert np.allclose(alt2["gamma"], want, rtol=1e-12)
    assert np.array_equal(alt2["k_gamma"], _bf16(alt2["gamma"]))
    # the signs follow the moved residual: most agree, the ones that change are where
    # the projection of the moved coordinate's column shifts p across zero
    assert (alt2["k_sign"] != rec["k_sign"]).any()


# --------------------------------------------------------------------------- #
# Bypass decode over plain bf16 pages                                            #
# --------------------------------------------------------------------------- #

def _bf16_pages(rng, B, Hkv, G, d, P, lens, nb_extra=2):
    lens = np.asarray(lens, np.int32)
    npg = (lens + P - 1) // P
    nb = int(npg.sum()) + nb_extra
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((B, max(int(npg.max()), 1)), -1, np.int32)
    st = 0
    for b in range(B):
        bt[b, : npg[b]] = perm[st: st + npg[b]]
        st += npg[b]
    kp = _bf16(rng.standard_normal((nb, Hkv, P, d)))
    vp = _bf16(rng.standard_normal((nb, Hkv, P, d)))
    q = _bf16(rng.standard_normal((B, Hkv * G, d)))
    return q, kp, vp, bt, lens


def test_bypass_decode_is_softmax_attention():
    """Against scipy's softmax over the gathered rows (a library routine) on tiny inputs."""
    from scipy.special import softmax
    rng = np.random.default_rng(41)
    B, Hkv, G, d, P = 3, 2, 3, 64, 16
    q, kp, vp, bt, lens = _bf16_pages(rng, B, Hkv, G, d, P, (37, 16, 5))
    sm = d ** -0.5
    out = O.decode_bf16(q, kp, vp, bt, lens, Hkv, P, sm)
    qd, kd, vd = O.bf16_to_double(q), O.bf16_to_double(kp), O.bf16_to_double(vp)
    for b in range(B):
        pos = np.arange(lens[b])
        blk, off = bt[b, pos // P], pos % P
        for h in range(Hkv * G):
            K = kd[blk, h // G, off]
            V = vd[blk, h // G, off]
            want = softmax(sm * (K @ qd[b, h])) @ V
            assert np.abs(out[b, h] - want).max() < 1e-12


def test_bypass_decode_special_cases():
    rng = np.random.default_rng(42)
    B, Hkv, G, d, P = 4, 1, 2, 32, 16
    q, kp, vp, bt, lens = _bf16_pages(rng, B, Hkv, G, d, P, (1, 0, 20, 20))
    kp[bt[2, 0], 0] = kp[bt[2, 0], 0, :1]  # identical keys on the first page of sequence 2
    kp[bt[2, 1], 0] = kp[bt[2, 0], 0, :1]
    q[3] = 0                                # zero query on sequence 3
    out = O.decode_bf16(q, kp, vp, bt, lens, Hkv, P, d ** -0.5)
    vd = O.bf16_to_double(vp)
    assert np.array_equal(out[0, 0], vd[bt[0, 0], 0, 0])   # one token: its value
    assert not out[1].any()                                  # no tokens: zeros
    rows = np.concatenate([vd[bt[2, 0], 0, :16], vd[bt[2, 1], 0, :4]])
    assert np.allclose(out[2, 0], rows.mean(0), atol=1e-12)  # identical keys: the mean value
    rows3 = np.concatenate([vd[bt[3, 0], 0, :16], vd[bt[3, 1], 0, :4]])
    assert np.allclose(out[3, 1], rows3.mean(0), atol=1e-12)  # zero query: the mean value



# --------------------------------------------------------------------------- #
# Values coded by the rotation and the Lloyd-Max codebook                        #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("vbits", [2, 3, 4])
def test_mse_values_codebook_distortion(vbits):
    """Rotated unit values scaled by sqrt(d) are ~N(0,1): the coding error per
    coordinate is the Lloyd-Max distortion of N(0,1) at v_bits (J. Max 1960), the
    stored norm is bf16(||v||), a zero value is an all-zero record."""
    d = 128
    ora = O.Oracle(d, 4, vbits, 32, seed=5, values="mse")
    rng = np.random.default_rng(50 + vbits)
    v = _bf16(rng.standard_normal((3000, d)) * np.exp(rng.standard_normal((3000, 1))))
    v[7] = 0
    rec = ora.compress_rows(v=v)
    vc = ora.params()["v_centroids"]
    codes = np.stack([O.unpack(r, d, vbits) for r in rec["v_code"]])
    rows = np.arange(len(v)) != 7
    mse = np.mean((rec["vz"][rows] - vc[codes[rows]]) ** 2)
    assert abs(mse - MAX_MSE[vbits]) < 0.05 * MAX_MSE[vbits]
    assert np.array_equal(rec["v_meta"][:, 0], _bf16(np.linalg.norm(O.bf16_to_double(v), axis=1)))
    assert not rec["v_code"][7].any() and rec["v_meta"][7, 0] == 0


@pytest.mark.parametrize("d,rotation", [(128, 0), (256, 1)])
def test_mse_values_dequant_rotates_back_to_the_codebook(d, rotation):
    """V~ read back by dequant_slots, rotated by Pi and scaled by sqrt(d) / n16, is
    exactly the value centroids of the codes numpy decodes from the raw bytes."""
    from parity import read_records
    P, Hkv, T = 16, 2, 40
    ora = O.Oracle(d, 3, 3, 32, seed=12, rotation=rotation, values="mse")
    rng = np.random.default_rng(12)
    k = _bf16(rng.standard_normal((T, Hkv, d)))
    v = _bf16(rng.standard_normal((T, Hkv, d)) * 2.0)
    nb = T // P + 2
    slots = rng.permutation(nb * P)[:T].astype(np.int64)
    kc, vc = ora.compress_kv(k, v, slots, P, nb)
    _, V = ora.dequant_slots(kc, vc, P, Hkv, slots)
    rec = read_records(kc, vc, ora.geometry(P), d, 3, 3, 32, P, Hkv, slots, vmse=True)
    n16 = O.bf16_to_double(rec["v_norm"])
    u = np.einsum("ij,thj->thi", ora.params()["Pi"], V) * math.sqrt(d) / n16[..., None]
    assert np.abs(u - ora.params()["v_centroids"][rec["v_code"]]).max() < 1e-10


def test_mse_values_decode_matches_dense_attention():
    """Decode accumulating the MSE values in the rotated space and rotating back
    once equals dense softmax attention over the dequantised K~, V~ (numpy), and
    equals the original-space decode."""
    ora = O.Oracle(128, 3, 3, 32, seed=4, values="mse")
    rng = np.random.default_rng(4)
    B, Hkv, G, d, P = 2, 2, 2, 128, 16
    lens = np.array([37, 5], np.int32)
    npg = (lens + P - 1) // P
    nb = int(npg.sum()) + 1
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((B, int(npg.max())), -1, np.int32)
    st = 0
    for b in range(B):
        bt[b, : npg[b]] = perm[st: st + npg[b]]
        st += npg[b]
    T = int(lens.sum())
    k = _bf16(rng.standard_normal((T, Hkv, d)))
    v = _bf16(rng.standard_normal((T, Hkv, d)))
    slots = np.concatenate([bt[b, np.arange(lens[b]) // P].astype(np.int64) * P + np.arange(lens[b]) % P
                            for b in range(B)])
    kc, vc = ora.compress_kv(k, v, slots, P, nb)
    q = _bf16(rng.standard_normal((B, Hkv * G, d)))
    c = dict(q=q, kc=kc, vc=vc, bt=bt, lens=lens, P=P, Hkv=Hkv, slots=slots, d=d)
    sm = d ** -0.5
    ref = _numpy_attention(ora, c, sm)
    for mode in (0, 1):
        out = ora.decode(q, kc, vc, bt, lens, Hkv, P, sm, mode=mode)
        assert np.abs(out - ref).max() < 1e-10 * max(1.0, np.abs(ref).max())


# --------------------------------------------------------------------------- #
# Prefill: causal attention of the last positions of every sequence              #
# --------------------------------------------------------------------------- #

def test_prefill_is_causal_dense_attention():
    """Against numpy causal softmax attention over the dequantised K~, V~; the last
    query token equals the decode of the whole sequence; a query at position 0
    returns the first value."""
    ora, c = _tiny_case(lens=(37, 16, 5))
    d, Hkv, P = c["d"], c["Hkv"], c["P"]
    B, Tq, Hq = 3, 5, c["q"].shape[1]
    G = Hq // Hkv
    rng = np.random.default_rng(77)
    q = _bf16(rng.standard_normal((B, Tq, Hq, d)))
    sm = d ** -0.5
    out = ora.prefill(q, c["kc"], c["vc"], c["bt"], c["lens"], Hkv, P, sm)
    qd = O.bf16_to_double(q)
    for b in range(B):
        L = int(c["lens"][b])
        pos = np.arange(L)
        slots = c["bt"][b, pos // P].astype(np.int64) * P + pos % P
        K, V = ora.dequant_slots(c["kc"], c["vc"], P, Hkv, slots)
        for i in range(Tq):
            p_i = L - Tq + i
            for h in range(Hq):
                if p_i < 0:
                    assert not out[b, i, h].any()
                    continue
                s = sm * K[: p_i + 1, h // G] @ qd[b, i, h]
                w = np.exp(s - s.max())
                want = (w / w.sum()) @ V[: p_i + 1, h // G]
                assert np.abs(out[b, i, h] - want).max() < 1e-10 * max(1.0, np.abs(want).max())
    dec = ora.decode(q[:, -1], c["kc"], c["vc"], c["bt"], c["lens"], Hkv, P, sm)
    assert np.array_equal(out[:, -1], dec)
    # sequence 2 has 5 tokens and 5 queries: its first query sits at position 0
    _, V = ora.dequant_slots(c["kc"], c["vc"], P, Hkv, [int(c["bt"][2, 0]) * P])
    for h in range(Hq):
        assert np.allclose(out[2, 0, h], V[0, h // G], atol=1e-12)
