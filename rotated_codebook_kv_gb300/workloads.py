"""Seeded synthetic workloads for KV-cache compression and compressed-KV decode.

This module only draws inputs: shapes, value distributions, outlier structure,
page assignment and slot mappings.  It holds none of the codec's arithmetic,
so both the CUDA library's tests and the CPU oracle can take their inputs from
it.  Every draw comes from one ``torch.Generator`` seeded per (workload, layer).

Workloads (value distributions follow the pages' shapes; inputs are synthetic):

* ``pr1_tiny``       -- 1 sequence of 512 tokens, 2 KV / 4 query heads, d=128;
  K, V ~ N(0,1) with 4 random channels per KV head scaled x8 (same channels
  for K and V); K 3-bit codebook + QJL, V 4-bit, group 32; page size 16.
* ``compress_only``  -- 262,144 tokens x 8 KV heads, d=128; per-channel
  log-normal scale exp(0.5 N(0,1)) drawn per (K/V, head, channel); K 4-bit
  (no QJL), V 4-bit group 64; page size 16; slot mapping a random permutation
  of all 16,384 x 16 slots.
* ``paged_decode``   -- batch 32, 32 query / 8 KV heads, d=128, sequence
  lengths uniform in [1024, 8192]; K 3-bit + QJL, V 2-bit group 32; page 16.
* ``wide_head_decode`` -- batch 8, 16 query / 8 KV heads, d=256, 32,768 tokens
  each; K 4-bit, V 4-bit group 64; page 32; 2% of tokens (one Bernoulli draw
  per token, shared by heads, K and V) scaled x4.
* ``long_context_mixed`` -- 8 layers, (k_bits, v_bits) per layer drawn from
  {(4,4),(4,3),(3,3),(3,2),(2,2)}; batch 4, 64 query / 8 KV heads, d=128,
  131,072 tokens each, page 16, V group 32.

Decode workloads place each sequence's pages on physical blocks taken in order
from one random permutation of all blocks; the slot of token position ``t`` of
sequence ``b`` is ``block_table[b, t // P] * P + t % P``.  Unused block-table
entries hold -1.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional, Tuple

import torch

LAYER_BIT_PAIRS = [(4, 4), (4, 3), (3, 3), (3, 2), (2, 2)]


@dataclass(frozen=True)
class Workload:
    name: str
    head_dim: int
    k_bits: int
    v_bits: int
    group: int
    page_size: int
    num_kv_heads: int
    num_q_heads: int = 0          # 0: compress-only
    batch: int = 0                # decode sequences
    seq_len: int = 0              # fixed length (0: drawn)
    seq_len_range: Optional[Tuple[int, int]] = None
    num_tokens: int = 0           # compress-only token count
    num_blocks: int = 0           # compress-only pool size
    layers: int = 1
    layer_bits: Tuple[Tuple[int, int], ...] = field(default_factory=tuple)
    structure: str = "gaussian"   # gaussian | channel_x8 | channel_lognormal | token_x4
    seed: int = 0

    @property
    def decode(self) -> bool:
        return self.num_q_heads > 0

    def for_layer(self, layer: int) -> "Workload":
        """The single-layer workload of ``layer`` (bits from ``layer_bits``)."""
        if not self.layer_bits:
            return self
        kb, vb = self.layer_bits[layer]
        return replace(self, k_bits=kb, v_bits=vb, layers=1, layer_bits=(), name=f"{self.name}.L{layer}")

    def codec_seed(self, layer: int = 0) -> int:
        """Seed of the rotation / QJL matrices: workload seed plus layer."""
        return self.seed + layer


def _draw_layer_bits(n_layers: int, seed: int) -> Tuple[Tuple[int, int], ...]:
    g = torch.Generator().manual_seed(seed)
    idx = torch.randint(0, len(LAYER_BIT_PAIRS), (n_layers,), generator=g)
    return tuple(LAYER_BIT_PAIRS[int(i)] for i in idx)


def pr1_tiny(seed: int = 0) -> Workload:
    return Workload("pr1_tiny", 128, 3, 4, 32, 16, num_kv_heads=2, num_q_heads=4, batch=1, seq_len=512,
                    structure="channel_x8", seed=seed)


def compress_only(seed: int = 0) -> Workload:
    return Workload("compress_only", 128, 4, 4, 64, 16, num_kv_heads=8, num_tokens=262144, num_blocks=16384,
                    structure="channel_lognormal", seed=seed)


def paged_decode(seed: int = 0) -> Workload:
    return Workload("paged_decode", 128, 3, 2, 32, 16, num_kv_heads=8, num_q_heads=32, batch=32,
                    seq_len_range=(1024, 8192), seed=seed)


def wide_head_decode(seed: int = 0) -> Workload:
    return Workload("wide_head_decode", 256, 4, 4, 64, 32, num_kv_heads=8, num_q_heads=16, batch=8,
                    seq_len=32768, structure="token_x4", seed=seed)


def long_context_mixed(seed: int = 0) -> Workload:
    return Workload("long_context_mixed", 128, 4, 4, 32, 16, num_kv_heads=8, num_q_heads=64, batch=4,
                    seq_len=131072, layers=8, layer_bits=_draw_layer_bits(8, seed), seed=seed)


WORKLOADS = {
    "pr1_tiny": pr1_tiny,
    "compress_only": compress_only,
    "paged_decode": paged_decode,
    "wide_head_decode": wide_head_decode,
    "long_context_mixed": long_context_mixed,
}


def scaled(w: Workload, **kw) -> Workload:
    """A smaller or altered copy (for tests): any field may be overridden."""
    return replace(w, **kw)


@dataclass
class Batch:
    """One layer's inputs.  Tensors live on the generation device."""
    k: torch.Tensor              # [T, Hkv, d] bf16
    v: torch.Tensor              # [T, Hkv, d] bf16
    slot_mapping: torch.Tensor   # [T] int64
    num_blocks: int
    q: Optional[torch.Tensor] = None            # [B, Hq, d] bf16
    block_table: Optional[torch.Tensor] = None  # [B, max_blocks] int32
    seq_lens: Optional[torch.Tensor] = None     # [B] int32
    sm_scale: float = 0.0

    @property
    def num_tokens(self) -> int:
        return self.k.shape[0]


def _gen(device, seed: int) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


def generate(w: Workload, layer: int = 0, device="cpu") -> Batch:
    """Draw the inputs of layer ``layer`` of workload ``w`` on ``device``."""
    device = torch.device(device)
    g = _gen(device, w.seed * 1000 + layer)
    d, H, P = w.head_dim, w.num_kv_heads, w.page_size

    # --- sequence lengths and page placement ---------------------------------
    if w.decode:
        if w.seq_len_range is not None:
            lo, hi = w.seq_len_range
            seq_lens = torch.randint(lo, hi + 1, (w.batch,), generator=g, device=device).to(torch.int32)
        else:
            seq_lens = torch.full((w.batch,), w.seq_len, dtype=torch.int32, device=device)
        npages = (seq_lens.to(torch.int64) + P - 1) // P
        num_blocks = int(npages.sum())
        max_blocks = int(npages.max()) if w.batch else 0
        perm = torch.randperm(num_blocks, generator=g, device=device).to(torch.int32)
        block_table = torch.full((w.batch, max(max_blocks, 1)), -1, dtype=torch.int32, device=device)
        starts = torch.cumsum(npages, 0) - npages
        col = torch.arange(max(max_blocks, 1), device=device)
        valid = col[None, :] < npages[:, None]
        src = (starts[:, None] + col[None, :]).clamp(max=max(num_blocks - 1, 0))
        block_table = torch.where(valid, perm[src], block_table)
        # token order: sequences concatenated, positions ascending
        T = int(seq_lens.to(torch.int64).sum())
        b_of_t = torch.repeat_interleave(torch.arange(w.batch, device=device), seq_lens.to(torch.int64))
        tok_start = torch.cumsum(seq_lens.to(torch.int64), 0) - seq_lens.to(torch.int64)
        pos = torch.arange(T, device=device) - tok_start[b_of_t]
        slot_mapping = block_table[b_of_t, pos // P].to(torch.int64) * P + pos % P
    else:
        T, num_blocks = w.num_tokens, w.num_blocks
        seq_lens = block_table = None
        slot_mapping = torch.randperm(num_blocks * P, generator=g, device=device)[:T].to(torch.int64)

    # --- K and V values --------------------------------------------------------
    k = torch.randn(T, H, d, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(T, H, d, generator=g, device=device, dtype=torch.float32)
    if w.structure == "channel_x8":
        ch = torch.stack([torch.randperm(d, generator=g, device=device)[:4] for _ in range(H)])  # [H, 4]
        s = torch.ones(H, d, device=device)
        s.scatter_(1, ch, 8.0)
        k *= s
        v *= s
    elif w.structure == "channel_lognormal":
        sk = torch.exp(0.5 * torch.randn(H, d, generator=g, device=device))
        sv = torch.exp(0.5 * torch.randn(H, d, generator=g, device=device))
        k *= sk
        v *= sv
    elif w.structure == "token_x4":
        out = (torch.rand(T, generator=g, device=device) < 0.02).to(torch.float32) * 3.0 + 1.0
        k *= out[:, None, None]
        v *= out[:, None, None]
    k = k.to(torch.bfloat16)
    v = v.to(torch.bfloat16)

    if not w.decode:
        return Batch(k, v, slot_mapping, num_blocks)
    q = torch.randn(w.batch, w.num_q_heads, d, generator=g, device=device).to(torch.bfloat16)
    return Batch(k, v, slot_mapping, num_blocks, q=q, block_table=block_table, seq_lens=seq_lens,
                 sm_scale=float(d) ** -0.5)


def as_u16(t: torch.Tensor):
    """Raw bit pattern of a bf16 tensor as a numpy uint16 array (host copy)."""
    import numpy as np
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
