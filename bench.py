#!/usr/bin/env python3
"""Benchmark: compress the full context, then decode one token, for every layer of
the long-context mixed-bit workload (8 layers; per-layer (k_bits, v_bits) drawn
from {(4,4),(4,3),(3,3),(3,2),(2,2)}; batch 4, 64 query / 8 KV heads, d=128,
131,072 tokens per sequence, page size 16, V group 32) on synthetic data.

One step = every hot-path call over one batch: for each layer, tq_compress_kv of
all 524,288 tokens x 8 KV heads, then tq_decode_attention of one query token per
sequence (3 launches).  Inputs (17 GB of bf16 K/V) exceed L2, and the order is
compress all layers then decode all layers, so each decode reads pages last
touched several GB of traffic earlier.

The printed value is whole-step algorithmic throughput in GB/s: bytes that must
move (K/V read, slots read, records written; records, queries, block tables
read and outputs written for decode) over the device time of a step.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference]
For N > 1 launch with torch.distributed.run; every rank runs its own copy of the
workload (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rotated_codebook_kv_gb300 import workloads as W  # noqa: E402

METRIC = "decode attn compressed-KV GB/s & % HBM roofline; compress Mtoken-heads/s"
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------- #
# Algorithmic bytes                                                             #
# --------------------------------------------------------------------------- #

def record_bytes(d, kb, vb, g, vmse=False):
    """Key and value record bytes per token-head (vmse: values as codes + a bf16 norm)."""
    qjl = kb <= 3
    k = d * kb // 8 + (d // 8 + 2 if qjl else 0) + 2
    v = d * vb // 8 + (2 if vmse else 4 * (d // g))
    return k, v


def compress_bytes(w, T, vmse=False):
    """Read K and V rows and the slot, write both records, per token-head."""
    k, v = record_bytes(w.head_dim, w.k_bits, w.v_bits, w.group, vmse)
    rows = T * w.num_kv_heads
    return rows * (4 * w.head_dim + k + v) + T * 8


def decode_bytes(w, seq_lens, max_blocks, vmse=False):
    k, v = record_bytes(w.head_dim, w.k_bits, w.v_bits, w.group, vmse)
    toks = int(sum(seq_lens))
    pages = sum((int(s) + w.page_size - 1) // w.page_size for s in seq_lens)
    qo = 2 * w.batch * w.num_q_heads * w.head_dim * 2
    return toks * w.num_kv_heads * (k + v) + qo + pages * 4 + w.batch * 4


# --------------------------------------------------------------------------- #
# Environment helpers                                                           #
# --------------------------------------------------------------------------- #

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        for key in ("hbm_gbs", "hbm_gbs_burst", "hbm_copy_gbs"):
            if key in peaks and isinstance(peaks[key], (int, float)):
                return float(peaks[key]), "measured"
            if key in peaks and isinstance(peaks[key], dict) and "value" in peaks[key]:
                return float(peaks[key]["value"]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s (burst) from MEASURED_PEAKS.json, else the recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, ValueError, KeyError, TypeError):
        return 1900.0


def committed_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current source."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            data = json.load(f)
        ent = data[kernel]
        src = open(os.path.join(ROOT, ent["source"]), "rb").read()
        if hashlib.sha256(src).hexdigest() != ent["source_sha256"]:
            return None
        return ent
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """Samples nvidia-smi clocks / throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "10"], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.window = None
        return self

    def mark(self, start):
        """Host time of the timed region's start / end: samples outside it are dropped."""
        now = time.time()
        if start:
            self.window = [now, None]
        elif self.window is not None:
            self.window[1] = now

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        if self.window is not None and self.window[1] is not None:
            inside = []
            for r in rows:
                try:
                    ts = datetime.datetime.strptime(r[9], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except (ValueError, IndexError):
                    continue
                if self.window[0] <= ts <= self.window[1]:
                    inside.append(r)
            if inside:
                rows = inside
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- #
# GPU arm                                                                        #
# --------------------------------------------------------------------------- #

class Layer:
    def __init__(self, w, layer, device, pinned_host=False):
        from rotated_codebook_kv_gb300 import Codec
        self.w = lw = w.for_layer(layer)
        self.codec = Codec(lw.head_dim, lw.k_bits, lw.v_bits, lw.group, lw.codec_seed(layer))
        b = W.generate(lw, layer=layer, device=device)
        self.b = b
        self.kc, self.vc = self.codec.alloc_cache(b.num_blocks, lw.num_kv_heads, lw.page_size, device=device)
        self.maxb = b.block_table.shape[1]
        self.splits = self.codec.decode_splits(lw.batch, lw.num_kv_heads, self.maxb, lw.page_size)
        self.ws = self.codec.workspace(lw.batch, lw.num_q_heads, self.splits, device=device)
        self.out = torch.empty_like(b.q)
        self.T = b.num_tokens
        self.seq_lens = b.seq_lens.cpu().tolist()
        self.c_bytes = compress_bytes(lw, self.T)
        self.d_bytes = decode_bytes(lw, self.seq_lens, self.maxb)
        self.host = None
        if pinned_host:
            self.host = {n: getattr(b, n).cpu().pin_memory() for n in
                         ("k", "v", "slot_mapping", "q", "block_table", "seq_lens")}
            self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()

    def compress(self, stream):
        lw, b = self.w, self.b
        self.codec.compress_kv(b.k, b.v, b.slot_mapping, self.kc, self.vc, lw.page_size, b.num_blocks, stream=stream)

    def decode(self, stream):
        lw, b = self.w, self.b
        self.codec.decode_attention(b.q, self.kc, self.vc, b.block_table, b.seq_lens, lw.num_kv_heads, lw.page_size,
                                    b.num_blocks, b.sm_scale, splits=self.splits, workspace=self.ws, out=self.out,
                                    stream=stream)

    def h2d(self, stream):
        with torch.cuda.stream(stream):
            for n, t in self.host.items():
                getattr(self.b, n).copy_(t, non_blocking=True)
        return sum(t.numel() * t.element_size() for t in self.host.values())

    def h2d_split(self, streams):
        """The same copies on two copy streams: keys on the first, values and the small
        tensors on the second, so that two copy engines run at once."""
        for n, t in self.host.items():
            with torch.cuda.stream(streams[0] if n == "k" else streams[1]):
                getattr(self.b, n).copy_(t, non_blocking=True)
        return sum(t.numel() * t.element_size() for t in self.host.values())

    def d2h(self, stream):
        with torch.cuda.stream(stream):
            self.out_host.copy_(self.out, non_blocking=True)
        return self.out.numel() * self.out.element_size()


def run_gpu(args, rank, world, local_rank):
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = rank_workload(rank, args.layers, args.batch)
    layers = [Layer(w, l, dev, pinned_host=not args.no_e2e) for l in range(w.layers)]
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def events(n):
        return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]

    c_ev = [events(len(layers)) for _ in range(args.steps)]
    d_ev = [events(len(layers)) for _ in range(args.steps)]

    def step(s=None):
        for i, L in enumerate(layers):
            if s is not None:
                c_ev[s][i][0].record(stream)
            L.compress(stream)
            if s is not None:
                c_ev[s][i][1].record(stream)
        for i, L in enumerate(layers):
            if s is not None:
                d_ev[s][i][0].record(stream)
            L.decode(stream)
            if s is not None:
                d_ev[s][i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for L in layers:
        if L.codec.get_status(stream) != 0:
            raise RuntimeError("device status bits set during warm-up")

    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize()
        clocks.mark(True)
        t0.record(stream)
        for s_ in range(args.steps):
            step(s_)
        t1.record(stream)
        torch.cuda.synchronize()
        clocks.mark(False)
    c_ms = [sum(c_ev[s_][i][0].elapsed_time(c_ev[s_][i][1]) for s_ in range(args.steps)) for i in range(len(layers))]
    d_ms = [sum(d_ev[s_][i][0].elapsed_time(d_ev[s_][i][1]) for s_ in range(args.steps)) for i in range(len(layers))]
    elapsed = t0.elapsed_time(t1) / args.steps
    elapsed = max_over_ranks(elapsed, world)
    clk = clocks.summary()

    step_bytes = sum(L.c_bytes + L.d_bytes for L in layers)
    value = aggregate_value(step_bytes, elapsed, world)
    c_bytes = sum(L.c_bytes for L in layers)
    d_bytes = sum(L.d_bytes for L in layers)
    c_time = sum(c_ms) / args.steps * 1e-3
    d_time = sum(d_ms) / args.steps * 1e-3
    rows = sum(L.T * L.w.num_kv_heads for L in layers)
    peak, peak_kind = measured_peak()
    c_gbs = c_bytes / c_time / 1e9
    d_gbs = d_bytes / d_time / 1e9
    traffic = committed_traffic("compress_kernel")
    # per layer: tq_compress_kv is one launch, two at head dim 128 without QJL (the
    # keys-only tensor-core pass, then the value kernel); tq_decode_attention is three
    launches = args.steps * sum((2 if (L.w.head_dim == 128 and L.w.k_bits == 4) else 1) + 3 for L in layers)

    # ---- end to end: host buffers, copies inside the timed region ------------
    # The next layer's inputs are copied on two copy streams while this layer is
    # compressed; a layer's buffers are refilled only after its decode of the
    # previous step.  Every copy and kernel lies between the two events on `stream`.
    e2e = None
    if not args.no_e2e:
        cps = [torch.cuda.Stream(device=dev) for _ in range(2)]
        dec_done = [None] * len(layers)

        def e2e_step():
            h2d = d2h = 0
            for i, L in enumerate(layers):
                for s in cps:
                    if dec_done[i] is not None:
                        s.wait_event(dec_done[i])
                h2d += L.h2d_split(cps)
                for s in cps:
                    ev = torch.cuda.Event()
                    ev.record(s)
                    stream.wait_event(ev)
                L.compress(stream)
            for i, L in enumerate(layers):
                L.decode(stream)
                d2h += L.d2h(stream)
                dec_done[i] = torch.cuda.Event()
                dec_done[i].record(stream)
            return h2d, d2h

        e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h2d = d2h = 0
        e0.record(stream)
        for s in cps:
            s.wait_event(e0)
        for _ in range(args.steps):
            h2d, d2h = e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
        e2e = {"value": round(world * step_bytes / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e_ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    for L in layers:
        if L.codec.get_status(stream) != 0:
            raise RuntimeError("device status bits set during the timed region")

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in, fp32 compute, packed u8 cache",
        "data": "synthetic (seeded N(0,1) bf16 K/V/q; random page placement)",
        "config": {
            "workload": "long_context_mixed",
            "layers": w.layers,
            "layer_bits": [list(p) for p in w.layer_bits],
            "batch": w.batch, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "seq_len": w.seq_len, "page_size": w.page_size, "v_group": w.group,
            "decode_splits": [L.splits for L in layers],
            "l2": "inputs larger than L2 (17 GB K/V per step); no flush",
        },
        "compress_mtoken_heads_per_s": round(world * rows / c_time / 1e6, 1),
        "compress_gbs": round(c_gbs, 1),
        "compress_frac": round(c_gbs / peak, 4),
        "decode_gbs": round(d_gbs, 1),
        "decode_frac": round(d_gbs / peak, 4),
        "decode_kv_tokens_per_s": round(world * sum(sum(L.seq_lens) * L.w.num_kv_heads for L in layers) / d_time, 1),
        "decode_query_tokens_per_s": round(world * w.batch * w.layers / d_time, 1),
        "roofline": {
            "bound": "hbm", "kernel": "compress_tc_kernel (tq_compress_kv; 4-bit layers: its keys-only form + compress_values_tc_kernel)",
            "achieved": round(c_gbs, 1), "peak": peak, "peak_kind": f"of {peak_kind}",
            "unit": "GB/s", "frac": round(c_gbs / peak, 4),
            "traffic": None if traffic is None else traffic.get("bytes_per_launch"),
            "algorithmic_bytes_per_launch": round(c_bytes / len(layers)),
        },
        "roofline_decode": {
            "bound": "hbm", "kernel": "qrot_kernel + decode_mma_kernel + combine_kernel (tq_decode_attention)",
            "achieved": round(d_gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(d_gbs / peak, 4),
            "algorithmic_bytes_per_call": round(d_bytes / len(layers)),
        },
        "clocks": clk,
        "gpu_launches": launches,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_per_config:
        line["per_config"] = per_config(dev, peak, args.config_reps)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds)
    return line


# --------------------------------------------------------------------------- #
# The other full-size workloads                                                 #
# --------------------------------------------------------------------------- #

L2_FLUSH_BYTES = 2 * 129 * 1024 * 1024  # twice the GB300's L2


def per_config(dev, peak, reps, only=None):
    """Compress-only, paged-decode and wide-head workloads at full size, each call
    timed alone with CUDA events on its stream after an L2 flush (a write of twice
    the L2 size outside the timed region), so no call reads its inputs from L2.
    Median over `reps` calls after two warm-up calls."""
    from rotated_codebook_kv_gb300 import Codec
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def timed(fn):
        ms = []
        for i in range(reps + 2):
            with torch.cuda.stream(stream):
                flush.fill_(i & 0xff)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            stream.synchronize()
            if i >= 2:
                ms.append(a.elapsed_time(b))
        return statistics.median(ms) * 1e-3

    out = {}
    for name, w, rot, vals in (("compress_only", W.compress_only(), 0, "group"),
                               ("paged_decode", W.paged_decode(), 0, "group"),
                               ("wide_head_decode", W.wide_head_decode(), 0, "group"),
                               ("wide_head_decode_hadamard", W.wide_head_decode(), 1, "group"),
                               ("paged_decode_mse_values", W.paged_decode(), 0, "mse")):
        if only is not None and name != only:
            continue
        b = W.generate(w, device=dev)
        codec = Codec(w.head_dim, w.k_bits, w.v_bits, w.group, w.codec_seed(), rotation=rot, values=vals)
        kc, vc = codec.alloc_cache(b.num_blocks, w.num_kv_heads, w.page_size, device=dev)
        T = b.num_tokens
        t_c = timed(lambda: codec.compress_kv(b.k, b.v, b.slot_mapping, kc, vc, w.page_size, b.num_blocks,
                                              stream=stream))
        cb = compress_bytes(w, T, vals == "mse")
        ent = {"compress_mtoken_heads_per_s": round(T * w.num_kv_heads / t_c / 1e6, 1),
               "compress_gbs": round(cb / t_c / 1e9, 1), "compress_frac": round(cb / t_c / 1e9 / peak, 4),
               "compress_us": round(t_c * 1e6, 1)}
        if w.decode:
            maxb = b.block_table.shape[1]
            splits = codec.decode_splits(w.batch, w.num_kv_heads, maxb, w.page_size)
            ws = codec.workspace(w.batch, w.num_q_heads, splits, device=dev)
            o = torch.empty_like(b.q)
            t_d = timed(lambda: codec.decode_attention(b.q, kc, vc, b.block_table, b.seq_lens, w.num_kv_heads,
                                                       w.page_size, b.num_blocks, b.sm_scale, splits=splits,
                                                       workspace=ws, out=o, stream=stream))
            lens = b.seq_lens.cpu().tolist()
            db = decode_bytes(w, lens, maxb, vals == "mse")
            ent.update({"decode_gbs": round(db / t_d / 1e9, 1), "decode_frac": round(db / t_d / 1e9 / peak, 4),
                        "decode_us": round(t_d * 1e6, 1), "decode_splits": splits,
                        "decode_kv_tokens_per_s": round(sum(lens) * w.num_kv_heads / t_d, 1),
                        "decode_query_tokens_per_s": round(w.batch / t_d, 1)})
        if name == "paged_decode":
            # dequantisation of the whole cache back to bf16 (tq_dequant_kv): every record
            # read once, K and V written in bf16
            ko = torch.empty_like(b.k)
            vo = torch.empty_like(b.v)
            t_q = timed(lambda: codec.dequant_kv(kc, vc, w.page_size, b.num_blocks, w.num_kv_heads, b.slot_mapping,
                                                 k_out=ko, v_out=vo, stream=stream))
            qb = T * w.num_kv_heads * (sum(record_bytes(w.head_dim, w.k_bits, w.v_bits, w.group)) + 4 * w.head_dim) + T * 8
            ent.update({"dequant_gbs": round(qb / t_q / 1e9, 1), "dequant_frac": round(qb / t_q / 1e9 / peak, 4),
                        "dequant_us": round(t_q * 1e6, 1),
                        "dequant_mtoken_heads_per_s": round(T * w.num_kv_heads / t_q / 1e6, 1)})
            del ko, vo
        if codec.get_status(stream) != 0:
            raise RuntimeError(f"device status bits set in the {name} workload")
        out[name] = ent
        del b, kc, vc, codec
        torch.cuda.empty_cache()
    # the bypass decode (plain bf16 pages, same skeleton) on the long-context and paged shapes:
    # the bandwidth control of the compressed decode
    for name, w in (("bypass_bf16_long_context", W.long_context_mixed().for_layer(0)),
                    ("bypass_bf16_paged_decode", W.paged_decode())):
        if only is not None and name != only:
            continue
        b = W.generate(w, device=dev)
        codec = Codec(w.head_dim, 4, 4, 32, 0)
        P, H, d = w.page_size, w.num_kv_heads, w.head_dim
        kp = torch.empty(b.num_blocks * H * P, d, dtype=torch.bfloat16, device=dev)
        vp = torch.empty_like(kp)
        sm = b.slot_mapping
        rows = (((sm // P) * H)[:, None] + torch.arange(H, device=dev)[None, :]) * P + (sm % P)[:, None]
        kp[rows.reshape(-1)] = b.k.reshape(-1, d)
        vp[rows.reshape(-1)] = b.v.reshape(-1, d)
        del b.k, b.v
        maxb = b.block_table.shape[1]
        splits = codec.decode_splits(w.batch, H, maxb, P)
        ws = codec.workspace(w.batch, w.num_q_heads, splits, device=dev)
        o = torch.empty_like(b.q)
        t_d = timed(lambda: codec.decode_attention_bf16(b.q, kp, vp, b.block_table, b.seq_lens, H, P, b.num_blocks,
                                                        b.sm_scale, splits=splits, workspace=ws, out=o,
                                                        stream=stream))
        lens = b.seq_lens.cpu().tolist()
        db = sum(lens) * H * 4 * d + 2 * w.batch * w.num_q_heads * d * 2 + \
            sum((x + P - 1) // P for x in lens) * 4 + w.batch * 4
        if codec.get_status(stream) != 0:
            raise RuntimeError(f"device status bits set in the {name} workload")
        out[name] = {"decode_gbs": round(db / t_d / 1e9, 1), "decode_frac": round(db / t_d / 1e9 / peak, 4),
                     "decode_us": round(t_d * 1e6, 1), "decode_splits": splits,
                     "decode_kv_tokens_per_s": round(sum(lens) * H / t_d, 1),
                     "bytes_per_token_head": 4 * d}
        del kp, vp, b, codec
        torch.cuda.empty_cache()
    # chunked prefill over the compressed cache: the last 64 positions of every sequence of
    # the paged workload attend causally to their compressed context
    if only is not None and only != "prefill_paged_decode_chunk64":
        return out
    w = W.paged_decode()
    b = W.generate(w, device=dev)
    codec = Codec(w.head_dim, w.k_bits, w.v_bits, w.group, w.codec_seed())
    kc, vc = codec.alloc_cache(b.num_blocks, w.num_kv_heads, w.page_size, device=dev)
    codec.compress_kv(b.k, b.v, b.slot_mapping, kc, vc, w.page_size, b.num_blocks, stream=stream)
    Tq = 64
    gq = torch.Generator(device=dev).manual_seed(5)
    q = torch.randn(w.batch, Tq, w.num_q_heads, w.head_dim, generator=gq, device=dev).to(torch.bfloat16)
    o = torch.empty_like(q)
    t_p = timed(lambda: codec.prefill_attention(q, kc, vc, b.block_table, b.seq_lens, w.num_kv_heads, w.page_size,
                                                b.num_blocks, b.sm_scale, out=o, stream=stream))
    lens = b.seq_lens.cpu().tolist()
    pairs = sum(sum(max(L - Tq + i + 1, 0) for i in range(Tq)) for L in lens) * w.num_q_heads
    flops = pairs * 4 * w.head_dim  # q.k and p.v per (query token, head, key token)
    tf_peak = measured_tensor_peak()
    if codec.get_status(stream) != 0:
        raise RuntimeError("device status bits set in the prefill workload")
    out["prefill_paged_decode_chunk64"] = {
        "prefill_us": round(t_p * 1e6, 1), "prefill_query_tokens_per_s": round(w.batch * Tq / t_p, 1),
        "attention_tflops": round(flops / t_p / 1e12, 2), "tensor_peak_tflops": tf_peak,
        "tensor_frac": round(flops / t_p / 1e12 / tf_peak, 4),
        "note": "useful attention math (4 d flops per query-head-key pair) over the measured bf16 peak"}
    del q, o, kc, vc, b, codec
    torch.cuda.empty_cache()
    out["timing"] = f"median of {reps} calls after 2 warm-up calls; L2 flushed before each call"
    if "wide_head_decode_hadamard" in out:
        out["wide_head_decode_hadamard"]["rotation"] = "randomized Hadamard (tq_init_ex)"
    if "paged_decode_mse_values" in out:
        out["paged_decode_mse_values"]["values"] = "rotation + Lloyd-Max codebook (tq_init_ex, TQ_VALUES_MSE)"
    return out


# --------------------------------------------------------------------------- #
# CPU oracle (baseline / reference arm)                                         #
# --------------------------------------------------------------------------- #

class OracleSample:
    """A bounded sample of the same workload: per layer, the first `tok` tokens of
    `nseq` sequences on the first `nkv` KV heads, compressed then decoded (one
    query token per sequence, G query heads per KV head) by the CPU oracle."""

    def __init__(self, w, tok=1024, nseq=4, nkv=4):
        import oracle as O
        self.O = O
        self.items = []
        self.bytes = 0
        self.rows = 0
        for layer in range(w.layers):
            lw = W.scaled(w.for_layer(layer), batch=nseq, seq_len=tok, num_kv_heads=nkv,
                          num_q_heads=nkv * (w.num_q_heads // w.num_kv_heads))
            b = W.generate(lw, layer=layer, device="cpu")
            ora = O.Oracle(lw.head_dim, lw.k_bits, lw.v_bits, lw.group, w.codec_seed(layer))
            self.items.append((lw, b, ora, W.as_u16(b.k), W.as_u16(b.v), W.as_u16(b.q),
                               b.slot_mapping.numpy(), b.block_table.numpy(), b.seq_lens.numpy()))
            self.bytes += compress_bytes(lw, b.num_tokens) + decode_bytes(lw, b.seq_lens.tolist(),
                                                                           b.block_table.shape[1])
            self.rows += b.num_tokens * nkv
        self.desc = (f"per layer x{w.layers}: {tok} tokens x {nseq} sequences x {nkv} KV heads compressed, "
                     f"then decoded with {w.num_q_heads // w.num_kv_heads} query heads per KV head")

    def run(self, nthreads=0):
        for lw, b, ora, k, v, q, sm, bt, sl in self.items:
            kc, vc = ora.compress_kv(k, v, sm, lw.page_size, b.num_blocks, nthreads=nthreads)
            ora.decode(q, kc, vc, bt, sl, lw.num_kv_heads, lw.page_size, b.sm_scale, mode=1, nthreads=nthreads)


def cpu_model():
    try:  # lscpu names Arm cores too ("Neoverse-V2"); /proc/cpuinfo does not on aarch64
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip().lower() == "model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(w, budget_s=12.0):
    s = OracleSample(w)
    cores = os.cpu_count() or 1
    t = time.perf_counter()
    s.run()
    one = time.perf_counter() - t
    reps = max(1, min(int(budget_s / max(one, 1e-3)), 50))
    t = time.perf_counter()
    for _ in range(reps):
        s.run()
    el = time.perf_counter() - t
    # one thread on the first layer of the sample, for the per-core rate
    one_layer = OracleSample(W.scaled(w, layers=1, layer_bits=w.layer_bits[:1]))
    t = time.perf_counter()
    one_layer.run(nthreads=1)
    el1 = time.perf_counter() - t
    return {"value": round(s.bytes * reps / el / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{s.desc}; {reps} repetitions, {el:.1f} s", "seconds": round(el, 2),
            "single_thread_gbs": round(one_layer.bytes / el1 / 1e9, 5),
            "single_thread_sample": f"layer 0 of the sample on one thread, {el1:.1f} s",
            "cpu_model": cpu_model()}


def run_reference(args):
    w = W.long_context_mixed(seed=0)
    s = OracleSample(w)
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        s.run()
    t = time.perf_counter()
    for _ in range(args.steps):
        s.run()
    el = (time.perf_counter() - t) / args.steps
    value = s.bytes / el / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "long_context_mixed", "layers": w.layers,
                   "layer_bits": [list(p) for p in w.layer_bits], "sample": s.desc},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": s.desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# --------------------------------------------------------------------------- #
# Distributed plumbing                                                           #
# --------------------------------------------------------------------------- #

def rank_workload(rank, layers=None, batch=None):
    """Every rank gets the same shapes and per-layer bits (those of seed 0); only the data seed differs.

    layers / batch shrink the workload for profiling captures only; the
    benchmark line itself always uses the full workload."""
    w = W.long_context_mixed(seed=0)
    kw = {"seed": rank}
    if layers:
        kw.update(layers=layers, layer_bits=w.layer_bits[:layers])
    if batch:
        kw.update(batch=batch)
    return W.scaled(w, **kw)


def aggregate_value(step_bytes, step_ms, world):
    """Whole-job GB/s: every rank moves step_bytes per step; the step takes the slowest rank's time."""
    return world * step_bytes / (step_ms * 1e-3) / 1e9


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["tq", "reference"], default="tq")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-per-config", action="store_true", help="skip the other full-size workloads")
    ap.add_argument("--config-reps", type=int, default=10)
    ap.add_argument("--only", default=None,
                    help="profiling only: run just this entry of the other full-size workloads (one timed call)")
    ap.add_argument("--layers", type=int, default=None, help="profiling only: first N layers")
    ap.add_argument("--batch", type=int, default=None, help="profiling only: fewer sequences")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)))
        return 0

    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.only:  # profiling: one workload's calls (two warm-up calls and one timed), no benchmark line
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        print(json.dumps(per_config(dev, measured_peak()[0], 1, only=args.only)))
        return 0
    line = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
