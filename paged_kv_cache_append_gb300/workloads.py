"""Seeded synthetic workloads for the paged KV hot path.

This module only draws inputs: block tables (seeded permutations of physical
page ids), per-row context lengths, and bf16 q / K / V values.  It holds none
of the method's arithmetic (no codec, no attention) and is shared by the
tests, the benchmark and the smoke check.

Five workloads follow the shapes of the Paged KV Context Store's use (P = 64,
1..8 concurrent sequences, GQA with 16-32 query heads):

* ``tiny_bf16``      1 sequence, 1 layer, frontier 200 (4 pages, the last
                     with 8 valid), 8 q / 2 kv heads, D 128, M = 8 pages in a
                     seeded random order; decode of 1 token.
* ``int8_decode``    INT8-G64, C = 8 rows, contexts uniform in [1, 4096]
                     after appending one token, 16 q / 2 kv heads, D 256,
                     8 layers, M = C * 64 shuffled pages; K/V ~ N(0, 1) with 1%
                     of the elements scaled by 20.
* ``fp8_shared``     FP8-E4M3FN-row256, C = 8 rows of 32768-token capacity
                     that share the first 16384 tokens' pages (optionally a
                     Fork at a mid-page frontier with a copied tail), frontiers
                     at random mid-page offsets near 32768, 16 q / 2 kv heads,
                     D 256, 16 layers, M = 2560.
* ``k8v4_long``      K8V4 (K FP8-row, V NVFP4-G16), C = 8 rows at 131072
                     tokens, 32 q / 4 kv heads, D 128, 16 layers, M = 16384;
                     decode T = 1 or verify T = 4.
* ``bf16_prefill``   BF16, 2 rows with a 2048-token chunk after a mid-page
                     prefix of 30657..30719 tokens, plus 6 decode rows at
                     8192 tokens, 16 q / 2 kv heads, D 256, 16 layers, M = 4096.

Lengths and permutations use ``numpy.random.default_rng(seed)``; values use a
``torch.Generator`` seeded from (workload seed, layer, stream id, row), on the
CPU by default or on a CUDA device when the caller asks (large pools).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

P = 64


@dataclass
class Workload:
    name: str
    profile: str
    num_layers: int
    Hq: int
    Hkv: int
    D: int
    S: int                      # max context per sequence
    C: int                      # max concurrency = table rows
    M: int                      # physical page groups
    tables: np.ndarray          # int32 [C, L]
    # decode rows --------------------------------------------------------
    table_rows: np.ndarray      # int32 [B]  table row of compact row b
    context: np.ndarray         # int32 [B]  tokens in the cache before the step
    T: int = 1                  # query tokens per decode row (appended, then attended)
    # chunked prefill rows (bf16_prefill) ----------------------------------
    prefill_rows: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    prefix_len: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    chunk_len: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    Tc: int = 0
    # shared prefix (fp8_shared): rows share tokens [0, shared_len) of row 0's
    # pages; when shared_len is mid-page the tail page is a private copy
    shared_len: int = 0
    scale: float = 0.0
    seed: int = 0
    outlier_p: float = 0.0
    outlier_mul: float = 1.0
    # V = (N(0, 1) with outliers + v_offset) * v_mul, for value-range cases
    v_offset: float = 0.0
    v_mul: float = 1.0

    @property
    def L(self) -> int:
        return -(-self.S // P)

    @property
    def B(self) -> int:
        return int(self.table_rows.shape[0])

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    # -- value streams -------------------------------------------------
    def _gen(self, layer: int, stream: int, row: int, device) -> torch.Generator:
        g = torch.Generator(device=device)
        g.manual_seed(((self.seed * 1_000_003 + layer) * 131 + stream) * 1_009 + row)
        return g

    def _normal(self, shape, layer, stream, row, outliers, device, value=False):
        g = self._gen(layer, stream, row, device)
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if outliers and self.outlier_p > 0:
            u = torch.rand(shape, generator=g, device=device)
            x = torch.where(u < self.outlier_p, x * self.outlier_mul, x)
        if value and (self.v_offset != 0.0 or self.v_mul != 1.0):
            x = (x + self.v_offset) * self.v_mul
        return x.to(torch.bfloat16)

    def context_kv(self, layer: int, row: int, n: int, device="cpu"):
        """bf16 (K, V) [n, Hkv, D] of the first n cached tokens of table row ``row``."""
        shape = (n, self.Hkv, self.D)
        return (self._normal(shape, layer, 1, row, True, device),
                self._normal(shape, layer, 2, row, True, device, value=True))

    def step_kv(self, layer: int, device="cpu"):
        """bf16 (K, V) [B, T, Hkv, D] of the tokens each decode row appends."""
        shape = (self.B, self.T, self.Hkv, self.D)
        return (self._normal(shape, layer, 3, 0, True, device),
                self._normal(shape, layer, 4, 0, True, device, value=True))

    def step_q(self, layer: int, device="cpu"):
        """bf16 q [B, T, Hq, D] of the decode rows."""
        return self._normal((self.B, self.T, self.Hq, self.D), layer, 5, 0, False, device)

    def chunk_kv(self, layer: int, device="cpu"):
        """bf16 (K, V) [Bp, Tc, Hkv, D] of the prefill chunk tokens."""
        shape = (len(self.prefill_rows), self.Tc, self.Hkv, self.D)
        return (self._normal(shape, layer, 6, 0, True, device),
                self._normal(shape, layer, 7, 0, True, device, value=True))

    def chunk_q(self, layer: int, device="cpu"):
        return self._normal((len(self.prefill_rows), self.Tc, self.Hq, self.D), layer, 8, 0, False, device)


def _perm(seed: int, M: int) -> np.ndarray:
    return np.random.default_rng(seed).permutation(M).astype(np.int32)


def tiny_bf16() -> Workload:
    tables = _perm(1, 8)[None, :]
    return Workload("tiny_bf16", "bf16", 1, 8, 2, 128, 512, 1, 8, tables,
                    table_rows=np.array([0], np.int32), context=np.array([199], np.int32),
                    scale=1 / math.sqrt(128), seed=1001)


def int8_decode(num_layers: int = 8, C: int = 8, S: int = 4096) -> Workload:
    L = -(-S // P)
    M = C * L
    rng = np.random.default_rng(2)
    tables = _perm(2, M).reshape(C, L)
    context = rng.integers(0, S, C).astype(np.int32)          # then +1 appended
    return Workload("int8_decode", "int8_g64", num_layers, 16, 2, 256, S, C, M, tables,
                    table_rows=np.arange(C, dtype=np.int32), context=context,
                    scale=1 / math.sqrt(256), seed=1002, outlier_p=0.01, outlier_mul=20.0)


def fp8_shared(num_layers: int = 16, C: int = 8, S: int = 32768, shared_len: int | None = None,
               M: int | None = None) -> Workload:
    """Shared prefix of S/2 tokens (16384 at S = 32768) unless given."""
    if shared_len is None:
        shared_len = S // 2
    L = -(-S // P)
    full = shared_len // P
    if M is None:
        M = 2560 if (S, C) == (32768, 8) else full + C * (L - full) + 8
    rng = np.random.default_rng(3)
    perm = _perm(3, M)
    tables = np.zeros((C, L), np.int32)
    tables[:, :full] = perm[:full]                            # shared immutable pages
    nxt = full
    for r in range(C):
        tables[r, full:] = perm[nxt:nxt + L - full]
        nxt += L - full
    assert nxt <= M
    F_end = S - P + rng.integers(1, P, C)                     # mid-page frontiers
    return Workload("fp8_shared", "fp8_row", num_layers, 16, 2, 256, S, C, M, tables,
                    table_rows=np.arange(C, dtype=np.int32),
                    context=(F_end - 1).astype(np.int32), shared_len=shared_len,
                    scale=1 / math.sqrt(256), seed=1003)


def k8v4_long(T: int = 1, num_layers: int = 16, C: int = 8, S: int = 131072) -> Workload:
    L = -(-S // P)
    M = C * L
    tables = _perm(4, M).reshape(C, L)
    return Workload("k8v4_long" if T == 1 else "k8v4_verify", "k8v4", num_layers, 32, 4, 128,
                    S, C, M, tables, table_rows=np.arange(C, dtype=np.int32),
                    context=np.full(C, S - T, np.int32), T=T,
                    scale=1 / math.sqrt(128), seed=1004)


def bf16_prefill(num_layers: int = 16, S: int = 32768, Tc: int = 2048, decode_ctx: int = 8192,
                 n_prefill: int = 2, n_decode: int = 6, profile: str = "bf16") -> Workload:
    """The chunked-prefill workload; `profile` other than bf16 gives the same
    shapes over quantized pages (same seeds, so the same bf16 inputs)."""
    C = n_prefill + n_decode
    L = -(-S // P)
    M = 4096 if (S, C) == (32768, 8) else C * L
    rng = np.random.default_rng(5)
    tables = _perm(5, M)[:C * L].reshape(C, L)
    r = rng.integers(1, P, n_prefill)
    prefix = (S - Tc - P + r).astype(np.int32)                # mid-page prefix
    name = "bf16_prefill" if profile == "bf16" else f"{profile.split('_')[0]}_prefill"
    return Workload(name, profile, num_layers, 16, 2, 256, S, C, M, tables,
                    table_rows=np.arange(n_prefill, C, dtype=np.int32),
                    context=np.full(n_decode, decode_ctx - 1, np.int32),
                    prefill_rows=np.arange(n_prefill, dtype=np.int32), prefix_len=prefix,
                    chunk_len=np.full(n_prefill, Tc, np.int32), Tc=Tc,
                    scale=1 / math.sqrt(256), seed=1005)


WORKLOADS = {"tiny_bf16": tiny_bf16, "int8_decode": int8_decode, "fp8_shared": fp8_shared,
             "k8v4_long": k8v4_long, "bf16_prefill": bf16_prefill}


def bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
