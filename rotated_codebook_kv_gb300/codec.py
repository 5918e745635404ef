"""Torch-facing convenience wrapper over the C ABI (argument marshalling only).

Tensors must already live on the CUDA device; this module only turns them into
pointers, sizes and the current stream and calls ``libtq.so``.  There is no CPU
path: a CPU tensor raises.
"""
from __future__ import annotations

import torch

from . import native

__all__ = ["Codec"]


def _ptr(t: torch.Tensor) -> int:
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device (the library has no CPU path)")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Codec:
    """One set of codec tables (Pi, S, codebook) on the current device."""

    def __init__(self, head_dim: int, k_bits: int, v_bits: int, group: int, seed: int = 0, rotation: int = 0,
                 values: str = "group"):
        """rotation: native.TQ_ROTATION_DENSE (Haar) or native.TQ_ROTATION_HADAMARD;
        values: "group" (per-group scale / zero) or "mse" (rotation + Lloyd-Max codebook)."""
        self.head_dim, self.k_bits, self.v_bits, self.group, self.seed = head_dim, k_bits, v_bits, group, seed
        self.qjl = k_bits <= 3
        self.rotation = rotation
        self.values = values
        flags = (native.TQ_ROTATION_HADAMARD if rotation == native.TQ_ROTATION_HADAMARD else 0) | \
            (native.TQ_VALUES_MSE if values == "mse" else 0)
        self.handle = native.tq_init_ex(head_dim, k_bits, v_bits, group, seed, flags)

    def close(self):
        if getattr(self, "handle", None):
            native.tq_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- layout -----------------------------------------------------------------
    def cache_layout(self, page_size: int):
        return native.tq_cache_layout(self.handle, page_size)

    def alloc_cache(self, num_blocks: int, num_kv_heads: int, page_size: int, device="cuda", fill: int = 0):
        kpb, vpb = self.cache_layout(page_size)
        kc = torch.full((num_blocks * num_kv_heads * kpb,), fill, dtype=torch.uint8, device=device)
        vc = torch.full((num_blocks * num_kv_heads * vpb,), fill, dtype=torch.uint8, device=device)
        return kc, vc

    # ---- calls ------------------------------------------------------------------
    def compress_kv(self, k, v, slot_mapping, k_cache, v_cache, page_size: int, num_blocks: int, stream=None):
        T, H, d = k.shape
        assert v.shape == k.shape and d == self.head_dim and k.dtype == torch.bfloat16
        assert k.stride(2) == 1 and k.stride(1) == d and v.stride(2) == 1 and v.stride(1) == d
        native.tq_compress_kv(self.handle, _ptr(k), _ptr(v), T, H, k.stride(0), v.stride(0), _ptr(slot_mapping),
                              _ptr(k_cache), _ptr(v_cache), page_size, num_blocks, _stream(stream))

    def dequant_kv(self, k_cache, v_cache, page_size: int, num_blocks: int, num_kv_heads: int, slots,
                   k_out=None, v_out=None, stream=None):
        T = slots.numel()
        shape = (T, num_kv_heads, self.head_dim)
        if k_out is None:
            k_out = torch.zeros(shape, dtype=torch.bfloat16, device=slots.device)
        if v_out is None:
            v_out = torch.zeros(shape, dtype=torch.bfloat16, device=slots.device)
        native.tq_dequant_kv(self.handle, _ptr(k_cache), _ptr(v_cache), page_size, num_blocks, num_kv_heads,
                             _ptr(slots), T, _ptr(k_out), _ptr(v_out), _stream(stream))
        return k_out, v_out

    def decode_splits(self, batch: int, num_kv_heads: int, max_blocks_per_seq: int, page_size: int) -> int:
        return native.tq_decode_splits(self.handle, batch, num_kv_heads, max_blocks_per_seq, page_size)

    def workspace(self, batch: int, num_q_heads: int, splits: int, device="cuda"):
        n = native.tq_decode_workspace_bytes(self.handle, batch, num_q_heads, splits)
        return torch.empty(n, dtype=torch.uint8, device=device)

    def decode_attention(self, q, k_cache, v_cache, block_table, seq_lens, num_kv_heads: int, page_size: int,
                         num_blocks: int, sm_scale: float, splits: int = 0, workspace=None, out=None, stream=None):
        B, Hq, d = q.shape
        assert d == self.head_dim and q.dtype == torch.bfloat16 and q.is_contiguous()
        maxb = block_table.shape[1]
        if splits == 0:
            splits = self.decode_splits(B, num_kv_heads, maxb, page_size)
        if workspace is None:
            workspace = self.workspace(B, Hq, splits, device=q.device)
        if out is None:
            out = torch.empty_like(q)
        native.tq_decode_attention(self.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                   _ptr(seq_lens), B, Hq, num_kv_heads, page_size, maxb, num_blocks, float(sm_scale),
                                   splits, _ptr(workspace), workspace.numel(), _ptr(out), _stream(stream))
        return out

    def set_wait_limit(self, cycles: int):
        native.tq_set_wait_limit(self.handle, cycles)

    def prefill_attention(self, q, k_cache, v_cache, block_table, seq_lens, num_kv_heads: int, page_size: int,
                          num_blocks: int, sm_scale: float, splits: int = 0, workspace=None, out=None, stream=None):
        """Causal attention of the last q.shape[1] positions of every sequence over its compressed cache.

        q: [B, Tq, Hq, d] bf16; returns [B, Tq, Hq, d] bf16."""
        B, Tq, Hq, d = q.shape
        assert d == self.head_dim and q.dtype == torch.bfloat16 and q.is_contiguous()
        maxb = block_table.shape[1]
        if splits == 0:
            splits = native.tq_prefill_splits(self.handle, B, Tq, Hq, num_kv_heads, maxb, page_size)
        if workspace is None:
            workspace = self.workspace(B * Tq, Hq, splits, device=q.device)
        if out is None:
            out = torch.empty_like(q)
        native.tq_prefill_attention(self.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                    _ptr(seq_lens), B, Tq, Hq, num_kv_heads, page_size, maxb, num_blocks,
                                    float(sm_scale), splits, _ptr(workspace), workspace.numel(), _ptr(out),
                                    _stream(stream))
        return out

    def decode_attention_bf16(self, q, k_pool, v_pool, block_table, seq_lens, num_kv_heads: int, page_size: int,
                              num_blocks: int, sm_scale: float, splits: int = 0, workspace=None, out=None,
                              stream=None):
        """Bypass decode over plain bf16 pools [num_blocks][num_kv_heads][page_size][head_dim]."""
        B, Hq, d = q.shape
        assert d == self.head_dim and q.dtype == torch.bfloat16 and q.is_contiguous()
        assert k_pool.dtype == torch.bfloat16 and v_pool.dtype == torch.bfloat16
        maxb = block_table.shape[1]
        if splits == 0:
            splits = self.decode_splits(B, num_kv_heads, maxb, page_size)
        if workspace is None:
            workspace = self.workspace(B, Hq, splits, device=q.device)
        if out is None:
            out = torch.empty_like(q)
        native.tq_decode_attention_bf16(self.handle, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                        _ptr(seq_lens), B, Hq, num_kv_heads, page_size, maxb, num_blocks,
                                        float(sm_scale), splits, _ptr(workspace), workspace.numel(), _ptr(out),
                                        _stream(stream))
        return out

    def get_status(self, stream=None) -> int:
        return native.tq_get_status(self.handle, _stream(stream))

    def export_params(self):
        import numpy as np
        d, L = self.head_dim, 1 << self.k_bits
        Pi = np.zeros((d, d), np.float32)
        S = np.zeros((d, d), np.float32)
        c = np.zeros(L, np.float32)
        t = np.zeros(L - 1, np.float32)
        native.tq_export_params(self.handle, Pi.ctypes.data, S.ctypes.data, c.ctypes.data, t.ctypes.data)
        return {"Pi": Pi, "S": S, "centroids": c, "thresholds": t}
