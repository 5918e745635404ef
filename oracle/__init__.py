"""Double-precision CPU oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
in ``rotated_codebook_kv_gb300``; the C source ``tq_oracle.c`` documents which
passage of the method's description each step follows.

bf16 and fp16 values cross this interface as raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

# The oracle is compiled without FMA contraction or fast-math so that it gives
# the same doubles on x86-64 and aarch64 hosts.
_CFLAGS = ["-O2", "-fPIC", "-shared", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile ``tq_oracle.c`` into ``_build/liboracle.so`` (gcc) if stale."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        u8p, u16p, i32p, i64p, u64p, dp = (P(ctypes.c_uint8), P(ctypes.c_uint16), P(ctypes.c_int32),
                                           P(ctypes.c_int64), P(ctypes.c_uint64), P(ctypes.c_double))
        vp = ctypes.c_void_p
        sig = {
            "tq_or_splitmix64": (None, [ctypes.c_uint64, ctypes.c_int64, u64p]),
            "tq_or_gaussians": (None, [ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, dp]),
            "tq_or_rotation": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint64, dp]),
            "tq_or_qjl_matrix": (None, [ctypes.c_int, ctypes.c_uint64, dp]),
            "tq_or_codebook": (ctypes.c_int, [ctypes.c_int, dp, dp]),
            "tq_or_bf16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
            "tq_or_bf16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
            "tq_or_f16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
            "tq_or_f16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
            "tq_or_create": (vp, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64]),
            "tq_or_create2": (vp, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
                                   ctypes.c_uint64]),
            "tq_or_create3": (vp, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
                                   ctypes.c_uint64, ctypes.c_int]),
            "tq_or_hadamard_rotation": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint64, dp]),
            "tq_or_destroy": (None, [vp]),
            "tq_or_get_params": (None, [vp, dp, dp, dp, dp]),
            "tq_or_geometry": (None, [vp, ctypes.c_int, i64p]),
            "tq_or_pack": (None, [u8p, ctypes.c_int, ctypes.c_int, u8p]),
            "tq_or_unpack": (None, [u8p, ctypes.c_int, ctypes.c_int, u8p]),
            "tq_or_compress_rows": (None, [vp, u16p, u16p, ctypes.c_int64, u8p, u8p, u16p, u16p, u8p, u16p,
                                           dp, dp, dp, dp, dp, ctypes.c_int]),
            "tq_or_compress_kv": (ctypes.c_int64, [vp, u16p, u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
                                                   ctypes.c_int64, i64p, u8p, u8p, ctypes.c_int, ctypes.c_int64,
                                                   ctypes.c_int]),
            "tq_or_dequant_slots": (None, [vp, u8p, u8p, ctypes.c_int, ctypes.c_int, i64p, ctypes.c_int64, dp, dp]),
            "tq_or_key_qjl_given_codes": (None, [vp, u16p, u8p, ctypes.c_int64, u8p, u16p, dp, dp]),
            "tq_or_decode_bf16": (None, [u16p, u16p, u16p, i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, dp]),
            "tq_or_decode": (None, [vp, u16p, u8p, u8p, i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, i32p,
                                    ctypes.c_int64, dp, ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


# --------------------------------------------------------------------------- #
# Module-level primitives                                                      #
# --------------------------------------------------------------------------- #

def splitmix64(state: int, n: int) -> np.ndarray:
    out = np.zeros(n, dtype=np.uint64)
    _load().tq_or_splitmix64(ctypes.c_uint64(state), n, _ptr(out, ctypes.c_uint64))
    return out


def gaussians(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.zeros(n, dtype=np.float64)
    _load().tq_or_gaussians(ctypes.c_uint64(seed), stream, n, _ptr(out, ctypes.c_double))
    return out


def rotation(d: int, seed: int) -> np.ndarray:
    out = np.zeros((d, d), dtype=np.float64)
    rc = _load().tq_or_rotation(d, ctypes.c_uint64(seed), _ptr(out, ctypes.c_double))
    assert rc == 0
    return out


def hadamard_rotation(d: int, seed: int) -> np.ndarray:
    out = np.zeros((d, d), dtype=np.float64)
    rc = _load().tq_or_hadamard_rotation(d, ctypes.c_uint64(seed), _ptr(out, ctypes.c_double))
    assert rc == 0
    return out


def qjl_matrix(d: int, seed: int) -> np.ndarray:
    out = np.zeros((d, d), dtype=np.float64)
    _load().tq_or_qjl_matrix(d, ctypes.c_uint64(seed), _ptr(out, ctypes.c_double))
    return out


def codebook(bits: int):
    """(centroids[2^b], thresholds[2^b - 1], iterations) of the N(0,1) Lloyd-Max quantiser."""
    L = 1 << bits
    c = np.zeros(L)
    t = np.zeros(max(L - 1, 1))
    it = _load().tq_or_codebook(bits, _ptr(c, ctypes.c_double), _ptr(t, ctypes.c_double))
    return c, t[: L - 1], it


def bf16_from_double(x) -> np.ndarray:
    f = _load().tq_or_bf16_from_double
    x = np.asarray(x, dtype=np.float64)
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def bf16_to_double(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f16_from_double(x) -> np.ndarray:
    f = _load().tq_or_f16_from_double
    x = np.asarray(x, dtype=np.float64)
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def f16_to_double(h) -> np.ndarray:
    f = _load().tq_or_f16_to_double
    h = np.asarray(h, dtype=np.uint16)
    return np.array([f(int(v)) for v in h.ravel()], dtype=np.float64).reshape(h.shape)


def pack(codes, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    n = codes.size
    out = np.zeros((n * bits + 7) // 8, dtype=np.uint8)
    _load().tq_or_pack(_ptr(codes, ctypes.c_uint8), n, bits, _ptr(out, ctypes.c_uint8))
    return out


def unpack(packed, n: int, bits: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros(n, dtype=np.uint8)
    _load().tq_or_unpack(_ptr(packed, ctypes.c_uint8), n, bits, _ptr(out, ctypes.c_uint8))
    return out


def decode_bf16(q, k_pool, v_pool, block_table, seq_lens, Hkv: int, page_size: int, sm_scale: float):
    """Softmax attention of one query token per sequence over plain bf16 pages.

    q: [B, Hq, d] bf16 bits; pools: [num_blocks, Hkv, P, d] bf16 bits.  Returns [B, Hq, d] doubles."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    B, Hq, d = q.shape
    kp = np.ascontiguousarray(k_pool, dtype=np.uint16)
    vp = np.ascontiguousarray(v_pool, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((B, Hq, d))
    _load().tq_or_decode_bf16(_ptr(q, ctypes.c_uint16), _ptr(kp, ctypes.c_uint16), _ptr(vp, ctypes.c_uint16),
                              _ptr(bt, ctypes.c_int32), _ptr(sl, ctypes.c_int32), B, Hq, Hkv, d, page_size,
                              bt.shape[1], float(sm_scale), _ptr(out, ctypes.c_double))
    return out


# --------------------------------------------------------------------------- #
# Codec object                                                                  #
# --------------------------------------------------------------------------- #

class Oracle:
    """Parameters (Pi, S, codebook) for one (head_dim, k_bits, v_bits, group, seed).

    QJL is on iff ``k_bits <= 3``.
    """

    ROTATION_DENSE, ROTATION_HADAMARD = 0, 1

    def __init__(self, head_dim: int, k_bits: int, v_bits: int, group: int, seed: int,
                 qjl_seed: int | None = None, rotation: int = 0, values: str = "group"):
        """values: "group" (per-group scale / zero) or "mse" (rotation + Lloyd-Max codebook)."""
        self._lib = _load()
        options = (1 if rotation == self.ROTATION_HADAMARD else 0) | (2 if values == "mse" else 0)
        # a separate S seed is only for Monte-Carlo checks of the QJL estimator
        self._h = self._lib.tq_or_create3(head_dim, k_bits, v_bits, group, ctypes.c_uint64(seed),
                                          ctypes.c_uint64(seed if qjl_seed is None else qjl_seed), options)
        self.rotation = rotation
        self.values = values
        if not self._h:
            raise ValueError("unsupported oracle parameters")
        self.d, self.k_bits, self.v_bits, self.group, self.seed = head_dim, k_bits, v_bits, group, seed
        self.qjl = k_bits <= 3

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.tq_or_destroy(h)
            self._h = None

    def params(self):
        d, L = self.d, 1 << self.k_bits
        Pi, S = np.zeros((d, d)), np.zeros((d, d))
        c, t = np.zeros(L), np.zeros(L - 1)
        self._lib.tq_or_get_params(self._h, _ptr(Pi, ctypes.c_double), _ptr(S, ctypes.c_double),
                                   _ptr(c, ctypes.c_double), _ptr(t, ctypes.c_double))
        out = {"Pi": Pi, "S": S, "centroids": c, "thresholds": t}
        if self.values == "mse":
            vc, vt, _ = codebook(self.v_bits)
            out.update(v_centroids=vc, v_thresholds=vt)
        return out

    def geometry(self, page_size: int) -> dict:
        s = np.zeros(6, dtype=np.int64)
        self._lib.tq_or_geometry(self._h, page_size, _ptr(s, ctypes.c_int64))
        keys = ["k_code", "k_sign", "v_code", "v_meta", "k_page", "v_page"]
        return {k: int(v) for k, v in zip(keys, s)}

    def compress_rows(self, k=None, v=None, nthreads: int = 0, diag: bool = True) -> dict:
        """Records of n rows (k, v: [n, d] uint16 bf16 bits) as separate fields."""
        ref = k if k is not None else v
        n = ref.shape[0]
        g = self.geometry(16)
        k = None if k is None else np.ascontiguousarray(k, dtype=np.uint16)
        v = None if v is None else np.ascontiguousarray(v, dtype=np.uint16)
        out = {
            "k_code": np.zeros((n, g["k_code"]), np.uint8),
            "k_sign": np.zeros((n, max(g["k_sign"], 1)), np.uint8),
            "k_norm": np.zeros(n, np.uint16),
            "k_gamma": np.zeros(n, np.uint16),
            "v_code": np.zeros((n, g["v_code"]), np.uint8),
            "v_meta": np.zeros((n, g["v_meta"] // 2), np.uint16),
        }
        if diag:
            out.update(z=np.zeros((n, self.d)), pg=np.zeros((n, self.d)), norm=np.zeros(n), gamma=np.zeros(n),
                       vz=np.zeros((n, self.d)))
        self._lib.tq_or_compress_rows(
            self._h, _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16), n,
            _ptr(out["k_code"], ctypes.c_uint8), _ptr(out["k_sign"], ctypes.c_uint8),
            _ptr(out["k_norm"], ctypes.c_uint16), _ptr(out["k_gamma"], ctypes.c_uint16),
            _ptr(out["v_code"], ctypes.c_uint8), _ptr(out["v_meta"], ctypes.c_uint16),
            _ptr(out.get("z"), ctypes.c_double), _ptr(out.get("pg"), ctypes.c_double),
            _ptr(out.get("norm"), ctypes.c_double), _ptr(out.get("gamma"), ctypes.c_double),
            _ptr(out.get("vz"), ctypes.c_double), nthreads)
        if not self.qjl:
            out["k_sign"] = out["k_sign"][:, :0]
        return out

    def compress_kv(self, k, v, slot_mapping, page_size: int, num_blocks: int,
                    k_cache=None, v_cache=None, nthreads: int = 0):
        """Write K, V ([T, Hkv, d] uint16) into paged pools; returns (k_cache, v_cache)."""
        k = np.ascontiguousarray(k, dtype=np.uint16)
        v = np.ascontiguousarray(v, dtype=np.uint16)
        T, Hkv, d = k.shape
        assert d == self.d
        g = self.geometry(page_size)
        if k_cache is None:
            k_cache = np.zeros(num_blocks * Hkv * g["k_page"], np.uint8)
        if v_cache is None:
            v_cache = np.zeros(num_blocks * Hkv * g["v_page"], np.uint8)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        self._lib.tq_or_compress_kv(self._h, _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16), T, Hkv,
                                    Hkv * d, Hkv * d, _ptr(sm, ctypes.c_int64), _ptr(k_cache, ctypes.c_uint8),
                                    _ptr(v_cache, ctypes.c_uint8), page_size, num_blocks, nthreads)
        return k_cache, v_cache

    def key_qjl_given_codes(self, k, codes):
        """QJL signs / gamma of key rows ([n, d] bf16 bits) for given codes ([n, d] uint8)."""
        k = np.ascontiguousarray(k, dtype=np.uint16)
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        n = k.shape[0]
        out = {"k_sign": np.zeros((n, self.d // 8), np.uint8), "k_gamma": np.zeros(n, np.uint16),
               "pg": np.zeros((n, self.d)), "gamma": np.zeros(n)}
        self._lib.tq_or_key_qjl_given_codes(self._h, _ptr(k, ctypes.c_uint16), _ptr(codes, ctypes.c_uint8), n,
                                            _ptr(out["k_sign"], ctypes.c_uint8), _ptr(out["k_gamma"], ctypes.c_uint16),
                                            _ptr(out["pg"], ctypes.c_double), _ptr(out["gamma"], ctypes.c_double))
        return out

    def prefill(self, q, k_cache, v_cache, block_table, seq_lens, Hkv: int, page_size: int, sm_scale: float,
                mode: int = 1, nthreads: int = 0):
        """Causal attention of the last Tq positions of every sequence ([B, Tq, Hq, d] bf16 bits).

        Query token i of sequence b sits at position p = seq_lens[b] - Tq + i and
        attends to positions 0..p: by definition that is the one-token attention of
        that query over the first p + 1 tokens, so each (b, i) is one decode row with
        sequence length max(p + 1, 0) and sequence b's block table.  Returns
        [B, Tq, Hq, d] doubles."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        B, Tq, Hq, d = q.shape
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.asarray(seq_lens, dtype=np.int64)
        lens = np.maximum(sl[:, None] - Tq + np.arange(Tq)[None, :] + 1, 0).astype(np.int32).reshape(-1)
        bt_rows = np.repeat(bt, Tq, axis=0)
        out = self.decode(q.reshape(B * Tq, Hq, d), k_cache, v_cache, bt_rows, lens, Hkv, page_size, sm_scale,
                          mode=mode, nthreads=nthreads)
        return out.reshape(B, Tq, Hq, d)

    def dequant_slots(self, k_cache, v_cache, page_size: int, Hkv: int, slots):
        """K~ (original space) and V~ as doubles, [n_slots, Hkv, d]."""
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        n = slots.size
        ko = np.zeros((n, Hkv, self.d))
        vo = np.zeros((n, Hkv, self.d))
        self._lib.tq_or_dequant_slots(self._h, _ptr(np.ascontiguousarray(k_cache), ctypes.c_uint8),
                                      _ptr(np.ascontiguousarray(v_cache), ctypes.c_uint8), page_size, Hkv,
                                      _ptr(slots, ctypes.c_int64), n, _ptr(ko, ctypes.c_double),
                                      _ptr(vo, ctypes.c_double))
        return ko, vo

    def decode(self, q, k_cache, v_cache, block_table, seq_lens, Hkv: int, page_size: int,
               sm_scale: float, mode: int = 1, jobs=None, nthreads: int = 0, out=None):
        """Attention output [B, Hq, d] (double) for one query token per sequence.

        mode 0 scores against K~ in the original space, mode 1 in the rotated
        space from the codes.  ``jobs``: optional [(b, kv_head), ...] subset.
        """
        q = np.ascontiguousarray(q, dtype=np.uint16)
        B, Hq, d = q.shape
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        if out is None:
            out = np.zeros((B, Hq, d))
        jb = None if jobs is None else np.ascontiguousarray(np.asarray(jobs, dtype=np.int32).reshape(-1, 2))
        self._lib.tq_or_decode(self._h, _ptr(q, ctypes.c_uint16), _ptr(np.ascontiguousarray(k_cache), ctypes.c_uint8),
                               _ptr(np.ascontiguousarray(v_cache), ctypes.c_uint8), _ptr(bt, ctypes.c_int32),
                               _ptr(sl, ctypes.c_int32), B, Hq, Hkv, page_size, bt.shape[1], float(sm_scale), mode,
                               _ptr(jb, ctypes.c_int32), 0 if jb is None else jb.shape[0],
                               _ptr(out, ctypes.c_double), nthreads)
        return out
