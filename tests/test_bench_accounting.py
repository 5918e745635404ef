"""The benchmark's algorithmic byte counts: record sizes per token-head and the
whole-launch totals of the five workloads, checked against figures worked out
from the record layouts by hand (key codes d b_k / 8 B, QJL signs d / 8 B, bf16
norm and gamma 2 B each; value codes d b_v / 8 B, an fp16 scale and zero per
group).  CPU only."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from rotated_codebook_kv_gb300 import workloads as W  # noqa: E402


@pytest.mark.parametrize("d,kb,vb,g,expect", [
    (128, 3, 4, 32, 148),    # tiny workload: 68 B key record (48 + 16 + 2 + 2), 80 B value record (64 + 16)
    (128, 4, 4, 64, 138),    # compress-only: 66 + 72
    (128, 3, 2, 32, 116),    # paged decode: 68 + 48
    (256, 4, 4, 64, 274),    # wide head: 130 + 144
    (128, 4, 3, 32, 130),    # long-context layer pairs
    (128, 3, 3, 32, 132),
    (128, 2, 2, 32, 100),
    (128, 4, 4, 32, 146),
])
def test_record_bytes_per_token_head(d, kb, vb, g, expect):
    k, v = bench.record_bytes(d, kb, vb, g)
    assert k + v == expect


def test_compress_only_launch_bytes():
    # 2,097,152 token-heads x (512 B read + 138 B records + 1 B of slot per token-head)
    w = W.compress_only()
    assert bench.compress_bytes(w, w.num_tokens) == 2_097_152 * 651 == 1_365_245_952


def test_decode_bytes_count_records_queries_and_tables():
    w = W.scaled(W.paged_decode(), batch=2, seq_len_range=None, seq_len=33)
    seq_lens = [33, 1]
    got = bench.decode_bytes(w, seq_lens, max_blocks=3)
    records = (33 + 1) * w.num_kv_heads * 116
    q_and_out = 2 * 2 * w.num_q_heads * 128 * 2
    table = (3 + 1) * 4 + 2 * 4   # block ids of the pages read, plus seq_lens
    assert got == records + q_and_out + table
