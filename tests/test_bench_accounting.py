"""The benchmark's algorithmic work per launch (the numerator of every roofline
fraction it prints), on the CPU: bench.Bench's accounting, fed the per-token
bytes of the oracle's plane schema (itself pinned to the page's D = 256 byte
table), reproduces the per-launch figures the measurements quote, and counts
the decode's bytes as the sum over rows of F_b x KV heads x bytes per token
head (shared pages once) plus q, out and lse."""

import numpy as np
import pytest

import bench
from oracle import layout


class _Pool:
    def __init__(self, w):
        self.bpt = layout.bytes_per_token_head(w.profile, w.D)

    def kv_bytes_per_token_head(self):
        return self.bpt


def _accounting(name):
    w = bench.make_workload(name, layers=1)
    b = object.__new__(bench.Bench)  # the accounting only; no device state
    b.w, b.B, b.fused, b.pool = w, w.B, True, _Pool(w)
    return w, b


@pytest.mark.parametrize("name,per_launch", [
    ("k8v4_long", 847_404_352),      # 8 rows x 131,073 tokens x 4 KV heads x 202 B + q/out/lse + append
    ("k8v4_verify", 847_869_184),
    ("int8_decode", 14_339_552),
    ("fp8_shared", 152_050_112),     # shared pages counted once (unique bytes)
])
def test_bytes_per_launch(name, per_launch):
    w, b = _accounting(name)
    assert b.bytes_roofline_launch() == per_launch


def test_decode_bytes_are_the_visible_kv_plus_q_out_lse():
    w, b = _accounting("k8v4_long")
    bpt = layout.bytes_per_token_head("k8v4", 128)
    assert bpt == 128 + 2 + 64 + 8  # K codes, K row scale, V codes (E2M1), V group scales
    F = (w.context + w.T).astype(np.int64)
    kv = int(F.sum()) * w.Hkv * bpt
    qo = w.B * w.T * w.Hq * (2 * w.D * 2 + 4)
    app = w.B * w.T * w.Hkv * (2 * w.D * 2 + bpt)
    assert b.bytes_decode_layer() == kv + qo
    assert b.bytes_append_layer() == app


def test_prefill_flops_are_the_pages_attention_pairs():
    """4 D Hq (prefix S + S (S + 1) / 2) per row: the "Resource scheduling
    and context cache" page's AttentionPairs with B = prefix, S = chunk."""
    w = bench.make_workload("bf16_prefill", layers=1)
    b = object.__new__(bench.Bench)
    b.w = w
    pairs = sum(int(p) * int(s) + int(s) * (int(s) + 1) // 2 for p, s in zip(w.prefix_len, w.chunk_len))
    assert b.flops_prefill_layer() == 4 * w.D * w.Hq * pairs == 2_129_196_482_560
