"""Pins of the oracle's primitives against values fixed outside the oracle.

* SplitMix64: published test vectors of the generator (Steele, Lea & Flood
  2014; the seed-1234567 vector is the one the Rosetta Code "Pseudo-random
  numbers/Splitmix64" task prints, the seed-0 vector is the reference C
  implementation's first outputs).
* Gaussian streams: moments and a Kolmogorov-Smirnov test against N(0,1).
* Rotation: orthogonality, and equality with LAPACK's QR (numpy) of the same
  Gaussian matrix after the same sign normalisation (the Q of a QR with a
  positive-diagonal R is unique).
* Codebook: Lloyd-Max fixed-point conditions evaluated by numerical
  integration (scipy.integrate.quad), symmetry, the 1-bit closed form
  +-sqrt(2/pi), and J. Max, "Quantizing for minimum distortion", IRE Trans.
  Inf. Theory 6(1), 1960, Table I (Gaussian, N = 4, 8, 16 levels).
* Rounding: bf16 / fp16 round-to-nearest-even against brute-force nearest
  representable values and against numpy's float64 -> float16 conversion.
* Packing: LSB-first round trips, and the byte patterns "four 2-bit values or
  two 4-bit values per byte" (0xsero/turboquant, "Value Compression").
"""
import math

import numpy as np
import pytest
from scipy import integrate, stats

import oracle as O


# --------------------------------------------------------------------------- #
# SplitMix64 / Gaussians                                                        #
# --------------------------------------------------------------------------- #

def test_splitmix64_published_vectors():
    assert [int(x) for x in O.splitmix64(1234567, 5)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]
    assert [int(x) for x in O.splitmix64(0, 3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_gaussian_stream_is_standard_normal():
    z = O.gaussians(7, 0, 200_000)
    assert abs(z.mean()) < 5 / math.sqrt(len(z))
    assert abs(z.var() - 1) < 5 * math.sqrt(2 / len(z))
    assert stats.kstest(z, "norm").pvalue > 1e-3
    # streams and seeds are distinct sequences
    assert not np.allclose(O.gaussians(7, 0, 64), O.gaussians(7, 1, 64))
    assert not np.allclose(O.gaussians(7, 0, 64), O.gaussians(8, 0, 64))
    # an odd count is a prefix of the even one
    assert np.array_equal(O.gaussians(3, 1, 9), O.gaussians(3, 1, 10)[:9])


# --------------------------------------------------------------------------- #
# Rotation                                                                       #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("d", [128, 256])
def test_rotation_is_orthogonal(d):
    Pi = O.rotation(d, 3)
    assert np.abs(Pi.T @ Pi - np.eye(d)).max() < 1e-12
    assert np.abs(Pi @ Pi.T - np.eye(d)).max() < 1e-12
    rng = np.random.default_rng(0)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    assert abs((Pi @ q) @ (Pi @ k) - q @ k) < 1e-10 * np.linalg.norm(q) * np.linalg.norm(k)


@pytest.mark.parametrize("d,seed", [(128, 0), (256, 5), (32, 11)])
def test_rotation_matches_lapack_qr(d, seed):
    G = O.gaussians(seed, 0, d * d).reshape(d, d)
    Q, R = np.linalg.qr(G)
    ref = Q * np.sign(np.diag(R))[None, :]
    assert np.abs(O.rotation(d, seed) - ref).max() < 1e-12


def test_rotation_entries_look_haar():
    d = 256
    Pi = O.rotation(d, 1)
    x = Pi.ravel() * math.sqrt(d)  # entries of a Haar matrix ~ N(0, 1/d)
    assert abs(x.mean()) < 0.02
    assert abs(x.var() - 1) < 0.02
    assert abs(abs(np.linalg.det(Pi)) - 1) < 1e-9


def test_qjl_matrix_is_stream_one():
    assert np.array_equal(O.qjl_matrix(128, 4).ravel(), O.gaussians(4, 1, 128 * 128))


# --------------------------------------------------------------------------- #
# Lloyd-Max codebook                                                            #
# --------------------------------------------------------------------------- #

def _cond_mean(a, b):
    num = integrate.quad(lambda x: x * stats.norm.pdf(x), a, b, epsabs=1e-14, epsrel=1e-13, limit=200)[0]
    den = integrate.quad(stats.norm.pdf, a, b, epsabs=1e-15, epsrel=1e-13, limit=200)[0]
    return num / den


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_lloyd_max_conditions(bits):
    c, t, it = O.codebook(bits)
    assert it > 0
    L = 1 << bits
    assert np.all(np.diff(c) > 0)
    # thresholds are midpoints of neighbouring centroids
    assert np.abs(t - 0.5 * (c[:-1] + c[1:])).max() < 1e-12
    # centroids are conditional means between thresholds (numerical integration)
    edges = np.concatenate([[-np.inf], t, [np.inf]])
    for i in range(L):
        assert abs(c[i] - _cond_mean(edges[i], edges[i + 1])) < 1e-10
    # symmetric about zero
    assert np.abs(c + c[::-1]).max() < 1e-12


def test_codebook_one_bit_closed_form():
    c, t, _ = O.codebook(1)
    assert np.allclose(c, [-math.sqrt(2 / math.pi), math.sqrt(2 / math.pi)], atol=1e-14)
    assert t.shape == (1,) and abs(t[0]) < 1e-15


# J. Max (1960), Table I: optimum Gaussian quantiser outputs / thresholds and
# mean-square error, positive half, 4 significant figures.
MAX_1960 = {
    2: dict(out=[0.4528, 1.510], thr=[0.0, 0.9816], mse=0.1175),
    3: dict(out=[0.2451, 0.7560, 1.344, 2.152], thr=[0.0, 0.5006, 1.050, 1.748], mse=0.03454),
    4: dict(out=[0.1284, 0.3881, 0.6568, 0.9424, 1.256, 1.618, 2.069, 2.733],
            thr=[0.0, 0.2582, 0.5224, 0.7996, 1.099, 1.437, 1.844, 2.401], mse=0.009497),
}


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codebook_matches_max_1960(bits):
    c, t, _ = O.codebook(bits)
    ref = MAX_1960[bits]
    L = 1 << bits
    pos_c = c[L // 2:]
    pos_t = t[L // 2 - 1:]
    assert np.allclose(pos_c, ref["out"], rtol=6e-4, atol=1e-4)
    assert np.allclose(pos_t, ref["thr"], rtol=6e-4, atol=1e-4)
    # distortion E[(X - Q(X))^2] by numerical integration
    edges = np.concatenate([[-np.inf], t, [np.inf]])
    mse = sum(integrate.quad(lambda x, ci=c[i]: (x - ci) ** 2 * stats.norm.pdf(x), edges[i], edges[i + 1],
                             epsabs=1e-14, limit=200)[0] for i in range(L))
    assert abs(mse - ref["mse"]) < 6e-4 * ref["mse"] + 1e-6


# --------------------------------------------------------------------------- #
# Rounding                                                                       #
# --------------------------------------------------------------------------- #

def _all_bf16_values():
    b = np.arange(0, 0x7F80, dtype=np.uint32)  # positive finite bf16 patterns
    return (b << 16).view(np.float32).astype(np.float64)


def test_bf16_rounding_is_nearest_even():
    vals = _all_bf16_values()
    rng = np.random.default_rng(1)
    idx = rng.integers(1, len(vals) - 2, 4000)
    lo, hi = vals[idx], vals[idx + 1]
    x = np.concatenate([lo + (hi - lo) * rng.random(4000), 0.5 * (lo + hi),  # random points and exact ties
                        -(lo + (hi - lo) * rng.random(4000))])
    got = O.bf16_to_double(O.bf16_from_double(x))
    ax = np.abs(x)
    j = np.searchsorted(vals, ax)  # vals[j-1] <= ax <= vals[j]
    a, b = vals[j - 1], vals[j]
    da, db = ax - a, b - ax
    even_a = ((np.arange(len(vals))[j - 1]) % 2) == 0
    ref = np.where(da < db, a, np.where(db < da, b, np.where(even_a, a, b))) * np.sign(x)
    assert np.array_equal(got, ref)
    # overflow, zero, subnormal
    assert O.bf16_from_double(1e39) == 0x7F80 and O.bf16_from_double(-0.0) == 0x8000
    assert O.bf16_to_double(O.bf16_from_double(2.0 ** -133)) == 2.0 ** -133


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-8, 5, 3000),
                        (np.arange(2048) + 0.5) * 2.0 ** -24,  # subnormal ties
                        np.array([65504.0, 65519.99, 65520.0, -7e4, 6.1e-5, 2.0 ** -14, 0.0])])
    with np.errstate(over="ignore"):  # values past the fp16 range round to infinity on purpose
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(O.f16_from_double(x), ref)
    assert np.array_equal(O.f16_to_double(ref), ref.view(np.float16).astype(np.float64))


# --------------------------------------------------------------------------- #
# Bit packing                                                                   #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("d", [128, 256])
def test_pack_roundtrip(bits, d):
    rng = np.random.default_rng(bits * d)
    codes = rng.integers(0, 1 << bits, d).astype(np.uint8)
    packed = O.pack(codes, bits)
    assert packed.size == d * bits // 8
    assert np.array_equal(O.unpack(packed, d, bits), codes)


def test_pack_byte_patterns():
    # four 2-bit values per byte, first value in the low bits
    assert list(O.pack([1, 2, 3, 0, 3, 3, 3, 3], 2)) == [0b00111001, 0xFF]
    # two 4-bit values per byte
    assert list(O.pack([0xA, 0x5, 0x1, 0xF], 4)) == [0x5A, 0xF1]
    # 3-bit: a bitstream of 8 codes per 3 bytes
    codes = [1, 2, 3, 4, 5, 6, 7, 0]
    bits = sum(c << (3 * i) for i, c in enumerate(codes))
    assert list(O.pack(codes, 3)) == [bits & 0xFF, (bits >> 8) & 0xFF, (bits >> 16) & 0xFF]
    # sign bits: bit i of byte i // 8
    assert list(O.pack([1, 0, 0, 0, 0, 0, 0, 1, 0, 1, 0, 0, 0, 0, 0, 0], 1)) == [0x81, 0x02]


# --------------------------------------------------------------------------- #
# Randomized Hadamard rotation                                                  #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("d,seed", [(128, 0), (256, 7), (64, 123)])
def test_hadamard_rotation_matches_scipy(d, seed):
    """Pi = H diag(s) / sqrt(d): H from scipy's Sylvester construction, s_j the sign
    of the top bit of the j-th raw output of SplitMix64 stream 0 (pinned above)."""
    from scipy.linalg import hadamard
    raw = O.splitmix64(seed ^ 0x9E3779B97F4A7C15, d)
    s = np.where(raw >> np.uint64(63), -1.0, 1.0)
    want = hadamard(d).astype(np.float64) * s[None, :] / np.sqrt(d)
    got = O.hadamard_rotation(d, seed)
    assert np.array_equal(got, want)
    assert np.abs(got.T @ got - np.eye(d)).max() < 1e-12


def test_hadamard_rotation_is_a_butterfly():
    """Pi x equals the fast Walsh-Hadamard butterfly of s * x, divided by sqrt(d)."""
    d, seed = 256, 3
    Pi = O.hadamard_rotation(d, seed)
    s = np.sign(Pi[0]) * 1.0  # row 0 of H is all ones: its signs are s
    rng = np.random.default_rng(0)
    x = rng.standard_normal(d)
    y = (s * x).copy()
    h = 1
    while h < d:
        for i in range(0, d, 2 * h):
            a, b = y[i:i + h].copy(), y[i + h:i + 2 * h].copy()
            y[i:i + h], y[i + h:i + 2 * h] = a + b, a - b
        h *= 2
    assert np.allclose(Pi @ x, y / np.sqrt(d), atol=1e-12)


def test_hadamard_codebook_distortion():
    """Keys rotated by the randomized Hadamard matrix have N(0,1)-like coordinates,
    so the Lloyd-Max distortion of the codebook (J. Max 1960) is met as with the
    Haar rotation."""
    d, bits = 128, 3
    ora = O.Oracle(d, bits, 4, 32, seed=1, rotation=1)
    rng = np.random.default_rng(3)
    k = O.bf16_from_double(rng.standard_normal((3000, d)))
    rec = ora.compress_rows(k=k)
    c = ora.params()["centroids"]
    codes = np.stack([O.unpack(r, d, bits) for r in rec["k_code"]])
    mse = np.mean((rec["z"] - c[codes]) ** 2)
    assert abs(mse - 0.03454) < 0.05 * 0.03454
