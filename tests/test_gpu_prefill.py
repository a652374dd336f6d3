"""GPU parity of the tcgen05 chunked prefill / replay attention against the
oracle, through the C ABI.  The chunk's K/V are appended first; every query
i < chunk_len[b] attends keys <= prefix_len[b] + i through the block table."""

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


def prefill_workload(Hkv, G, D, S, prefixes, chunks, Tc, seed, n_decode=0, layers=1, profile="bf16"):
    rng = np.random.default_rng(seed)
    C = len(prefixes) + n_decode
    L = -(-S // 64)
    M = C * L
    tables = rng.permutation(M).astype(np.int32).reshape(C, L)
    Bp = len(prefixes)
    return W.Workload("prefill_test", profile, layers, Hkv * G, Hkv, D, S, C, M, tables,
                      table_rows=np.arange(Bp, C, dtype=np.int32),
                      context=np.full(n_decode, 10, np.int32),
                      prefill_rows=np.arange(Bp, dtype=np.int32),
                      prefix_len=np.asarray(prefixes, np.int32), chunk_len=np.asarray(chunks, np.int32),
                      Tc=Tc, scale=1 / math.sqrt(D), seed=seed + 9000)


def run_prefill(w, layer=0, poison=False, sample_rows=None, order="page_major", kv_scale=1.0, q_scale=1.0,
                check=True):
    """Appends the chunk, runs the prefill on the GPU and (check) compares it
    with the oracle; returns the GPU (out, lse) on the CPU."""
    sc = Scenario(w, layers=(layer,), oracle=True, order=order)
    dev = "cuda"
    k, v = w.chunk_kv(layer)
    q = w.chunk_q(layer)
    if kv_scale != 1.0:  # chunk rows only: the prefix stays N(0, 1)
        k = (k.float() * kv_scale).to(torch.bfloat16)
        v = (v.float() * kv_scale).to(torch.bfloat16)
    if q_scale != 1.0:
        q = (q.float() * q_scale).to(torch.bfloat16)
    rows = torch.from_numpy(w.prefill_rows).to(dev)
    pre = torch.from_numpy(w.prefix_len).to(dev)
    chk = torch.from_numpy(w.chunk_len).to(dev)
    sc.gpu.append(layer, sc.tables_d, rows, pre, k.to(dev), v.to(dev), counts=chk)
    sc.orc.append(layer, w.tables, w.prefill_rows, w.prefix_len, bf16_to_bits(k), bf16_to_bits(v),
                  counts=w.chunk_len)
    if poison:  # bytes past each row's frontier in its last page: 0xFF (NaN bf16)
        for i, r in enumerate(w.prefill_rows):
            F = int(w.prefix_len[i] + w.chunk_len[i])
            if F % 64 == 0:
                continue
            g = int(w.tables[r, F // 64])
            for pi, plane in enumerate(sc.gpu.planes[layer]):
                rb = sc.gpu.row_bytes[pi]
                for hh in range(w.Hkv):
                    base = ((g * w.Hkv + hh) * 64) * rb
                    plane[base + (F % 64) * rb: base + 64 * rb] = 0xFF
    out, lse = sc.gpu.prefill(layer, q.to(dev), sc.tables_d, rows, pre, chk, w.scale)
    torch.cuda.synchronize()
    out, lse = out.cpu(), lse.cpu()
    if not check:
        return out, lse
    qf = OF.bf16_bits_to_f64(bf16_to_bits(q))
    for i, r in enumerate(w.prefill_rows):
        P0, Cn = int(w.prefix_len[i]), int(w.chunk_len[i])
        K, V = sc.orc.gather(layer, w.tables[r], P0 + Cn)
        toks = np.arange(Cn) if sample_rows is None else np.unique(np.clip(sample_rows, 0, Cn - 1))
        ref_o = np.zeros((len(toks), w.Hq, w.D))
        ref_l = np.zeros((len(toks), w.Hq))
        for n, t in enumerate(toks):
            o1, l1 = OA.decode(qf[i, t:t + 1], K, V, P0 + t + 1, w.scale)
            ref_o[n], ref_l[n] = o1[0], l1[0]
        compare_attention(out[i, toks], lse[i, toks], ref_o, ref_l)
        if Cn < w.Tc:   # rows past the chunk are not written
            assert torch.all(out[i, Cn:] == 0) and torch.all(torch.isneginf(lse[i, Cn:]))
    return out, lse


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [8, 1, 16])
def test_prefill_small(D, G):
    """Two rows: a mid-page prefix and a ragged chunk that spans several
    128-row tiles (and one row with an empty prefix)."""
    w = prefill_workload(2 if G < 16 else 1, G, D, 1024, prefixes=[133, 0], chunks=[300, 77], Tc=320,
                         seed=D + G)
    run_prefill(w)


def test_prefill_stale_tail_is_not_read():
    w = prefill_workload(2, 8, 256, 1024, prefixes=[100, 37], chunks=[45, 200], Tc=256, seed=5)
    run_prefill(w, poison=True)


def test_prefill_bf16_workload_sampled():
    """The BF16 chunked-prefill workload at full size, one layer: 2 rows, a
    2048-token chunk after a mid-page prefix of ~30.7k tokens, 16 q / 2 kv
    heads, D 256; sampled query rows are checked against the oracle."""
    w = W.bf16_prefill(num_layers=1)
    sample = np.array([0, 1, 63, 64, 127, 128, 1000, 1023, 2046, 2047])
    run_prefill(w, sample_rows=sample)


def test_prefill_negative_softmax_scale():
    """A negative softmax scale reverses the score order; the running maximum
    must follow the scaled scores, not the raw ones."""
    import dataclasses
    w = prefill_workload(2, 8, 128, 512, prefixes=[70, 0], chunks=[130, 64], Tc=192, seed=9)
    run_prefill(dataclasses.replace(w, scale=-w.scale))


@pytest.mark.parametrize("profile", ["fp8_row", "nvfp4_g16", "k8v4"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [8, 1, 16])
def test_quantized_prefill_small(profile, D, G):
    """Prefill over FP8-row, NVFP4-G16 and K8V4 pages: a mid-page prefix and a
    ragged chunk spanning several tiles, an empty prefix in the other row."""
    w = prefill_workload(2 if G < 16 else 1, G, D, 1024, prefixes=[133, 0], chunks=[300, 77], Tc=320,
                         seed=D + G + 3, profile=profile)
    run_prefill(w)


@pytest.mark.parametrize("profile", ["fp8_row", "k8v4"])
def test_quantized_prefill_stale_tail_is_not_read(profile):
    w = prefill_workload(2, 8, 256, 1024, prefixes=[100, 37], chunks=[45, 200], Tc=256, seed=15,
                         profile=profile)
    run_prefill(w, poison=True)


def test_quantized_prefill_negative_scale():
    import dataclasses
    w = prefill_workload(2, 8, 128, 512, prefixes=[70, 0], chunks=[130, 64], Tc=192, seed=19,
                         profile="k8v4")
    run_prefill(dataclasses.replace(w, scale=-w.scale))


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [8, 1, 16])
def test_int8_prefill_small(D, G):
    """INT8-G64 pages: dequantized to f16 once (code * group scale rounded to
    f16, the one inexact profile), within the attention tolerances."""
    w = prefill_workload(2 if G < 16 else 1, G, D, 1024, prefixes=[133, 0], chunks=[300, 77], Tc=320,
                         seed=D + G + 5, profile="int8_g64")
    run_prefill(w)


def test_int8_prefill_stale_tail_and_negative_scale():
    import dataclasses
    w = prefill_workload(2, 8, 256, 1024, prefixes=[100, 37], chunks=[45, 200], Tc=256, seed=17,
                         profile="int8_g64")
    run_prefill(w, poison=True)
    run_prefill(dataclasses.replace(w, scale=-w.scale))


def test_int8_prefill_power_of_two_scaling_is_exact():
    """Keys and values times 2^16 and queries times 2^-16 leave the INT8 codes
    unchanged and multiply the group scales by 2^16, so rows take the per-key
    shift (2^-3 before the f16 rounding).  Powers of two commute with every
    rounding on the way, so the output must be exactly 2^16 times the unscaled
    one (itself checked against the oracle) and the lse identical."""
    w = prefill_workload(2, 8, 128, 512, prefixes=[0, 0], chunks=[200, 130], Tc=256, seed=21,
                         profile="int8_g64")
    out0, lse0 = run_prefill(w)
    out1, lse1 = run_prefill(w, kv_scale=2.0 ** 16, q_scale=2.0 ** -16, check=False)
    assert torch.equal(out1.float(), out0.float() * 2.0 ** 16)
    assert torch.equal(lse1, lse0)


def test_int8_prefill_workload_sampled():
    """The chunked-prefill workload over INT8-G64 pages at full size, one layer."""
    w = W.bf16_prefill(num_layers=1, profile="int8_g64")
    sample = np.array([0, 1, 63, 64, 127, 128, 1000, 1023, 2046, 2047])
    run_prefill(w, sample_rows=sample)


def test_prefill_k8v4_workload_sampled():
    """The chunked-prefill workload over K8V4 pages at full size, one layer:
    2 rows, a 2048-token chunk after a mid-page prefix of ~30.7k tokens;
    sampled query rows against the oracle."""
    w = W.bf16_prefill(num_layers=1, profile="k8v4")
    sample = np.array([0, 1, 63, 64, 127, 128, 1000, 1023, 2046, 2047])
    run_prefill(w, sample_rows=sample)


@pytest.mark.parametrize("profile", ["bf16", "k8v4"])
def test_prefill_without_page_splits(profile):
    """152 tiles (one wave of 1-CTA-per-SM work) leave each tile whole
    (no partials); the other tests run split tiles."""
    w = prefill_workload(2, 8, 128, 1400, prefixes=[61], chunks=[1216], Tc=1216, seed=23, profile=profile)
    run_prefill(w, sample_rows=np.array([0, 15, 16, 600, 1215]))


@pytest.mark.parametrize("profile", ["bf16", "k8v4", "nvfp4_g16"])
def test_prefill_head_major_plane_order(profile):
    w = prefill_workload(2, 8, 256, 1024, prefixes=[133, 0], chunks=[300, 77], Tc=320, seed=29,
                         profile=profile)
    run_prefill(w, order="head_major")


@pytest.mark.parametrize("profile", ["bf16", "int8_g64", "fp8_row", "nvfp4_g16", "k8v4"])
def test_prefill_workspace_does_not_grow_with_the_context(profile):
    """The pages are dequantized inside the attention kernel, so the prefill
    workspace (split partials only) is the same for a 4096-token pool and a
    131072-token pool of the same heads, rows and chunk."""
    from paged_kv_cache_append_gb300 import nk
    sizes = []
    for S in (4096, 131072):
        L = S // 64
        pool = nk.Pool(profile, 1, 2, 256, S, 2, L)
        sizes.append(nk.nk_prefill_workspace_bytes(pool.handle, 2, 2048, 16))
        pool.close()
    assert sizes[0] == sizes[1], sizes


@pytest.mark.parametrize("profile", ["fp8_row", "k8v4"])
def test_fp8_key_prefill_with_an_outlier_query_channel(profile):
    """FP8-row keys go to the tensor cores as raw E4M3 codes, with each query
    row split into two E4M3 terms (hi + lo).  Elements below 2^-9 of the row's
    largest one are kept to an absolute 2^-17 of it, so a query whose dim 5 is
    30 times the others (small elements then fall below that edge) must still
    match the oracle within the attention tolerances."""
    w = prefill_workload(2, 8, 256, 1024, prefixes=[300, 61], chunks=[200, 150], Tc=256, seed=77,
                         profile=profile)
    sc = Scenario(w, layers=(0,), oracle=True)
    dev = "cuda"
    k, v = w.chunk_kv(0)
    q = w.chunk_q(0).float()
    q[..., 5] *= 30.0
    q = q.to(torch.bfloat16)
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
        toks = np.arange(0, Cn, 7)
        ref_o = np.zeros((len(toks), w.Hq, w.D))
        ref_l = np.zeros((len(toks), w.Hq))
        for n_, t in enumerate(toks):
            o1, l1 = OA.decode(qf[i, t:t + 1], K, V, P0 + t + 1, w.scale)
            ref_o[n_], ref_l[n_] = o1[0], l1[0]
        compare_attention(out[i, toks], lse[i, toks], ref_o, ref_l)
