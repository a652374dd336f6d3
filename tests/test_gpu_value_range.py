"""GPU parity when V is far from unit scale, through the C ABI.

V = (N(0, 1) with 1% outliers x20 + 0.5) * v_mul for v_mul from 2^-14 to
2^22 (where the outliers saturate the INT8-G64 and FP8-row binary16 scales at
65504), with a sharp softmax (scale 4 / sqrt(D)).  The codec rules fix what the
pages hold at every magnitude (binary16 scales go subnormal for small V and
saturate at 65504 for large INT8-G64 V; NVFP4 flushes to zero below its E4M3
range and saturates above it); the attention over those dequantized values
must then match the oracle's to the usual tolerance measured in units of
v_mul: |out - oracle| / v_mul <= 2e-2 + 2^-8 |oracle| / v_mul, LSE (which V
does not enter) to 1e-3.  A power-of-two v_mul scales a bf16 output exactly.
The BF16 prefill rounds each softmax weight to bf16 once (8 significant
bits: relative error <= 2^-8), so its error is also allowed
2^-8 sum_j p_j |v_j| / sum_j p_j, the oracle's attention over |V|.  (The
other paths keep 11 or more significant bits of each weight; with V's 20x
outliers and this sharp softmax that bound, not the fixed 2e-2, is what holds
for bf16 weights.)

Each case covers one kernel form: the warp-level decode (R = 8 query rows per
KV head, fused append), the tensor-core verify (R = 32: the transposed form at
head_dim 64 and 128, the other at 256) and the chunked prefill (BF16 and the
fused quantized prefill).
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import formats as OF
from paged_kv_cache_append_gb300 import workloads as W
from paged_kv_cache_append_gb300.workloads import bf16_to_bits
from tests.scenario import Scenario, compare_attention

pytestmark = pytest.mark.gpu

PROFILES = ["bf16", "int8_g64", "fp8_row", "nvfp4_g16", "k8v4"]
V_MULS = [2.0 ** -14, 2.0 ** -8, 2.0 ** 10, 2.0 ** 17, 2.0 ** 22]


def _workload(profile, D, G, T, seed, v_mul, contexts, S, prefill=None):
    rng = np.random.default_rng(seed)
    C = len(contexts) if prefill is None else len(prefill[0])
    L = -(-S // 64)
    M = C * L
    tables = rng.permutation(M).astype(np.int32).reshape(C, L)
    kw = dict(scale=4.0 / math.sqrt(D), seed=seed + 11000, outlier_p=0.01, outlier_mul=20.0,
              v_offset=0.5, v_mul=v_mul)
    if prefill is None:
        return W.Workload("value_range", profile, 1, 2 * G, 2, D, S, C, M, tables,
                          table_rows=np.arange(C, dtype=np.int32), context=np.asarray(contexts, np.int32),
                          T=T, **kw)
    prefixes, chunks, Tc = prefill
    return W.Workload("value_range_prefill", profile, 1, 2 * G, 2, D, S, C, M, tables,
                      table_rows=np.zeros(0, np.int32), context=np.zeros(0, np.int32),
                      prefill_rows=np.arange(C, dtype=np.int32), prefix_len=np.asarray(prefixes, np.int32),
                      chunk_len=np.asarray(chunks, np.int32), Tc=Tc, **kw)


def _compare(out, lse, ref_out, ref_lse, v_mul, abs_attn=None):
    # dividing by a power of two is exact in bf16 and in float64
    extra = None if abs_attn is None else 2.0 ** -8 * abs_attn / v_mul
    return compare_attention(out.float() / v_mul, lse, ref_out / v_mul, ref_lse, extra=extra)


def _decode(w, fused):
    sc = Scenario(w)
    q, out, lse, fr = sc.step(0, fused=fused)
    ref_out, ref_lse = sc.oracle_decode(0, q, fr)
    _compare(out, lse, ref_out, ref_lse, w.v_mul)


@pytest.mark.parametrize("v_mul", V_MULS)
@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("profile", PROFILES)
def test_decode_value_range(profile, D, v_mul):
    """Fused append + decode, one token per row, 8 query heads per KV head."""
    w = _workload(profile, D, 8, 1, seed=D + int(math.log2(v_mul)) + 40, v_mul=v_mul,
                  contexts=[0, 301, 699], S=700)
    _decode(w, fused=True)


@pytest.mark.parametrize("v_mul", V_MULS)
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("profile", ["fp8_row", "nvfp4_g16", "k8v4"])
def test_verify_value_range(profile, D, v_mul):
    """4-token verify with 8 query heads per KV head (32 rows per KV head)."""
    w = _workload(profile, D, 8, 4, seed=D + int(math.log2(v_mul)) + 80, v_mul=v_mul,
                  contexts=[0, 301, 696], S=700)
    _decode(w, fused=False)


@pytest.mark.parametrize("v_mul", V_MULS)
@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("profile", PROFILES)
def test_prefill_value_range(profile, D, v_mul):
    """A mid-page prefix and a ragged chunk of two 128-row tiles, plus a row
    with an empty prefix."""
    w = _workload(profile, D, 8, 1, seed=D + int(math.log2(v_mul)) + 120, v_mul=v_mul, contexts=None,
                  S=640, prefill=([133, 0], [180, 61], 192))
    sc = Scenario(w)
    dev = "cuda"
    k, v = w.chunk_kv(0)
    q = w.chunk_q(0)
    rows = torch.from_numpy(w.prefill_rows).to(dev)
    pre = torch.from_numpy(w.prefix_len).to(dev)
    chk = torch.from_numpy(w.chunk_len).to(dev)
    sc.gpu.append(0, sc.tables_d, rows, pre, k.to(dev), v.to(dev), counts=chk)
    sc.orc.append(0, w.tables, w.prefill_rows, w.prefix_len, bf16_to_bits(k), bf16_to_bits(v), counts=w.chunk_len)
    out, lse = sc.gpu.prefill(0, q.to(dev), sc.tables_d, rows, pre, chk, w.scale)
    torch.cuda.synchronize()
    out, lse = out.cpu(), lse.cpu()
    qf = OF.bf16_bits_to_f64(bf16_to_bits(q))
    for i, r in enumerate(w.prefill_rows):
        P0, Cn = int(w.prefix_len[i]), int(w.chunk_len[i])
        K, V = sc.orc.gather(0, w.tables[r], P0 + Cn)
        ref_o = np.zeros((Cn, w.Hq, w.D))
        ref_l = np.zeros((Cn, w.Hq))
        ref_a = np.zeros((Cn, w.Hq, w.D)) if profile == "bf16" else None
        for t in range(Cn):
            o1, l1 = OA.decode(qf[i, t:t + 1], K, V, P0 + t + 1, w.scale)
            ref_o[t], ref_l[t] = o1[0], l1[0]
            if ref_a is not None:
                ref_a[t] = OA.decode(qf[i, t:t + 1], K, np.abs(V), P0 + t + 1, w.scale)[0][0]
        _compare(out[i, :Cn], lse[i, :Cn], ref_o, ref_l, w.v_mul, ref_a)
