"""Helpers for comparing the CUDA library's cache bytes and outputs with the oracle.

Acceptance rules (the decision windows and the decode tolerance of the parity
criteria, with the readings of them that the tests apply):
* value codes, scales, zeros and the page layout: bit-exact;
* key codes: equal except where the oracle's z lies within 1e-6 (N(0,1)
  units) of a threshold; QJL signs: equal except where the oracle's |p_i| / gamma
  < 1e-6; each kind of mismatch < 1e-5 of its elements.  Where a code differs
  inside its window the row's signs and gamma are compared with the oracle's
  signs for the codes actually stored;
* bf16 norm / gamma: equal, or one bf16 ulp apart where the oracle's double lies
  within 1e-6 (relative) of a bf16 rounding midpoint;
* decode output (bf16): |gpu - oracle| <= 2e-3 + half a bf16 ulp of the oracle.
"""
from __future__ import annotations

import numpy as np

import oracle as O

CODE_WINDOW = 1e-6
SIGN_WINDOW = 1e-6
MISMATCH_FRACTION = 1e-5
DECODE_ATOL = 2e-3


def unpack_bits(b: np.ndarray, n: int, bits: int) -> np.ndarray:
    """[..., n*bits/8] uint8 LSB-first bitstreams -> [..., n] codes (numpy, independent of the oracle)."""
    flat = np.unpackbits(b, axis=-1, bitorder="little").reshape(*b.shape[:-1], n, bits).astype(np.uint32)
    return (flat << np.arange(bits, dtype=np.uint32)).sum(-1).astype(np.uint8)


def read_records(cache_k: np.ndarray, cache_v: np.ndarray, geo: dict, d: int, kb: int, vb: int, g: int, P: int,
                 Hkv: int, slots: np.ndarray, vmse: bool = False) -> dict:
    """Fields of the records at `slots` (all heads): arrays shaped [n_slots, Hkv, ...].

    vmse: values coded by the rotation and a Lloyd-Max codebook (a bf16 norm per
    token instead of a (scale, zero) pair per group)."""
    qjl = kb <= 3
    slots = np.asarray(slots, np.int64)
    blk, off = slots // P, slots % P
    rec = (blk[:, None] * Hkv + np.arange(Hkv)[None, :])  # [n, Hkv]
    kbase = rec * geo["k_page"]
    vbase = rec * geo["v_page"]

    def take(cache, base, width):
        idx = base[..., None] + np.arange(width)
        return cache[idx]

    kcb, ksb, vcb, vmb = geo["k_code"], geo["k_sign"], geo["v_code"], geo["v_meta"]
    o = off[:, None]
    out = {"k_code": unpack_bits(take(cache_k, kbase + o * kcb, kcb), d, kb)}
    norm_off = P * (kcb + ksb)
    out["k_norm"] = take(cache_k, kbase + norm_off + 2 * o, 2).view(np.uint16)[..., 0]
    if qjl:
        out["k_sign"] = unpack_bits(take(cache_k, kbase + P * kcb + o * ksb, ksb), d, 1)
        out["k_gamma"] = take(cache_k, kbase + norm_off + 2 * P + 2 * o, 2).view(np.uint16)[..., 0]
    out["v_code"] = unpack_bits(take(cache_v, vbase + o * vcb, vcb), d, vb)
    if vmse:
        out["v_norm"] = take(cache_v, vbase + P * vcb + 2 * o, 2).view(np.uint16)[..., 0]
    else:
        out["v_meta"] = take(cache_v, vbase + P * vcb + o * vmb, vmb).view(np.uint16).reshape(len(slots), Hkv, d // g, 2)
    return out


def _bf16_near_midpoint(x: np.ndarray, rel=1e-6) -> np.ndarray:
    """True where double x lies within rel (relative) of a bf16 rounding midpoint."""
    ax = np.abs(x).astype(np.float64)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    q = 2.0 ** (e - 7)  # bf16 spacing in [2^e, 2^(e+1))
    frac = ax / q - np.floor(ax / q)
    return np.abs(frac - 0.5) * q <= rel * ax


def _bf16_ulps(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    a = a_bits.astype(np.int64)
    b = b_bits.astype(np.int64)
    return np.abs(a - b)


def check_key_value_records(ora: "O.Oracle", k_rows: np.ndarray, v_rows: np.ndarray, gpu: dict, report: dict = None):
    """Compare GPU record fields (flattened to rows) against the oracle run on the same rows.

    k_rows, v_rows: [N, d] bf16 bits; gpu: dict of fields with leading dim N.
    """
    d, kb = ora.d, ora.k_bits
    N = k_rows.shape[0]
    ref = ora.compress_rows(k=k_rows, v=v_rows)
    vstats = {}
    if getattr(ora, "values", "group") == "mse":
        # ---- MSE values: codes within the threshold window, norm within one ulp at a midpoint
        ref_vcode = unpack_bits(ref["v_code"], d, ora.v_bits)
        vthr = ora.params()["v_thresholds"]
        vdist = np.abs(ref["vz"][..., None] - vthr[None, None, :]).min(-1)
        vmis = gpu["v_code"].reshape(N, d) != ref_vcode
        assert np.all(vdist[vmis] < CODE_WINDOW), f"value code mismatch outside window: {vdist[vmis].max()}"
        assert vmis.sum() <= MISMATCH_FRACTION * vmis.size, f"{vmis.sum()} value code mismatches of {vmis.size}"
        vn_ref = ref["v_meta"][:, 0]
        vdiff = _bf16_ulps(gpu["v_norm"].reshape(N), vn_ref)
        assert np.all(vdiff <= 1), "value norm off by more than one bf16 ulp"
        vexact = np.linalg.norm(O.bf16_to_double(v_rows), axis=1)
        assert np.all(_bf16_near_midpoint(vexact[vdiff > 0])), "value norm differs away from a rounding midpoint"
        vstats = {"value_code_mismatch": int(vmis.sum()), "value_norm_ulp": int((vdiff > 0).sum())}
    else:
        # ---- values: bit-exact
        ref_vcode = unpack_bits(ref["v_code"], d, ora.v_bits)
        assert np.array_equal(gpu["v_code"].reshape(N, d), ref_vcode), "value codes differ"
        assert np.array_equal(gpu["v_meta"].reshape(N, -1), ref["v_meta"]), "value scale/zero differ"
    # ---- key codes within the threshold window
    ref_code = unpack_bits(ref["k_code"], d, kb)
    gcode = gpu["k_code"].reshape(N, d)
    thr = ora.params()["thresholds"]
    zdist = np.abs(ref["z"][..., None] - thr[None, None, :]).min(-1)
    mism = gcode != ref_code
    assert np.all(zdist[mism] < CODE_WINDOW), f"code mismatch outside window: {zdist[mism].max()}"
    assert mism.sum() <= max(MISMATCH_FRACTION * mism.size, 0), f"{mism.sum()} code mismatches of {mism.size}"
    # ---- norm
    gn = gpu["k_norm"].reshape(N)
    diff = _bf16_ulps(gn, ref["k_norm"])
    bad = diff > 0
    assert np.all(diff <= 1), "norm off by more than one bf16 ulp"
    assert np.all(_bf16_near_midpoint(ref["norm"][bad])), "norm differs away from a rounding midpoint"
    stats = {"code_mismatch": int(mism.sum()), "elements": int(mism.size), "norm_ulp": int(bad.sum()), **vstats}
    if ora.qjl:
        rows_cm = np.nonzero(mism.any(1))[0]
        exp_sign = unpack_bits(ref["k_sign"], d, 1)
        exp_gam = ref["k_gamma"].copy()
        exp_gamd = ref["gamma"].copy()
        pg = ref["pg"].copy()
        if rows_cm.size:  # re-derive signs for the codes actually stored
            alt = ora.key_qjl_given_codes(k_rows[rows_cm], gcode[rows_cm])
            exp_sign[rows_cm] = unpack_bits(alt["k_sign"], d, 1)
            exp_gam[rows_cm] = alt["k_gamma"]
            exp_gamd[rows_cm] = alt["gamma"]
            pg[rows_cm] = alt["pg"]
        gs = gpu["k_sign"].reshape(N, d)
        smis = gs != exp_sign
        assert np.all(np.abs(pg[smis]) < SIGN_WINDOW), f"sign mismatch outside window: {np.abs(pg[smis]).max()}"
        assert smis.sum() <= MISMATCH_FRACTION * smis.size, f"{smis.sum()} sign mismatches of {smis.size}"
        gg = gpu["k_gamma"].reshape(N)
        gd = _bf16_ulps(gg, exp_gam)
        assert np.all(gd <= 1), "gamma off by more than one bf16 ulp"
        assert np.all(_bf16_near_midpoint(exp_gamd[gd > 0])), "gamma differs away from a rounding midpoint"
        stats.update(sign_mismatch=int(smis.sum()), gamma_ulp=int((gd > 0).sum()), rows_code_mismatch=int(rows_cm.size))
    if report is not None:
        report.update(stats)
    return stats


def check_decode(out_gpu_bf16: np.ndarray, ref: np.ndarray, atol: float = DECODE_ATOL):
    """|gpu - ref| <= atol + half a bf16 ulp of ref, elementwise."""
    g = O.bf16_to_double(out_gpu_bf16)
    ax = np.abs(ref)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    half_ulp = np.where(ax > 0, 2.0 ** (e - 8), 0.0)
    err = np.abs(g - ref)
    bound = atol + half_ulp
    if err.size and not np.all(err <= bound):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"decode error {err[i]:.3e} > bound {bound[i]:.3e} at {i} (gpu {g[i]:.6f}, "
                             f"ref {ref[i]:.6f}); {np.count_nonzero(err > bound)} of {err.size} outside")
    return float(err.max()) if err.size else 0.0
