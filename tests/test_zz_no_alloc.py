"""The decode entry point that allocates nothing.

Some callers cannot allocate device memory at all: code that runs inside an
allocator's own callbacks, runtimes whose device-memory budget is fixed at
start-up, and serving loops that must never block on the driver's allocator.
nk_paged_decode_attention_noalloc serves them: it keeps the split-K partials
in a static device array of the library instead of a caller workspace.

These tests call it through the C ABI twice in a row (the array keeps the
previous call's contents) and check each result against the oracle and
against what nk_paged_decode_attention returns for the same inputs, within
the parity tolerance of the other tests (against the other entry point,
whose output is itself bf16-rounded, half an ulp per side).  The shapes
cover a plan that fits the array, plans whose split count must be lowered to
fit
(with at least one split per row, with fewer slots than rows, and with the
tcgen05 kernel that takes several pieces per CTA), and a call too large for
the array, which is rejected before any launch.

This file is named to be collected last.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_append_gb300 import nk
from paged_kv_cache_append_gb300 import workloads as W
from tests.scenario import Scenario, compare_attention, oracle_row

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20      # NK_NOALLOC_SCRATCH_BYTES in include/nk.h


def _workload(profile, Hkv, G, D, T, contexts, seed, S=None):
    """B = len(contexts) rows with the given contexts before the step."""
    rng = np.random.default_rng(seed)
    C = len(contexts)
    S = S or -(-(max(contexts) + T) // 64) * 64
    L = -(-S // 64)
    M = C * L
    tables = rng.permutation(M).astype(np.int32).reshape(C, L)
    return W.Workload(f"noalloc_{profile}", profile, 1, Hkv * G, Hkv, D, S, C, M, tables,
                      table_rows=np.arange(C, dtype=np.int32),
                      context=np.asarray(contexts, np.int32), T=T, scale=1 / math.sqrt(D),
                      seed=seed + 9000, outlier_p=0.01, outlier_mul=20.0)


def _split_bytes(w):
    """Partial bytes of one split slot per (row, KV head): (m, l) + R x D fp32."""
    R = 8 * (-(-w.T * (w.Hq // w.Hkv) // 8))
    return w.B * w.Hkv * R * (8 + 4 * w.D)


def _noalloc(lib, sc, q, rows, fr, w):
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], q.shape[1], q.shape[2]), float("nan"), device=q.device)
    rc = lib.nk_paged_decode_attention_noalloc(
        q.data_ptr(), w.Hq, sc.gpu.handle, 0, sc.tables_d.data_ptr(), rows.data_ptr(),
        fr.data_ptr(), q.shape[0], q.shape[1], ctypes.c_float(w.scale), out.data_ptr(),
        lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.nk_last_error().decode()
    return out, lse


def _run(w, full_oracle=True, oracle_rows=None, lowered=False):
    lib = nk.load()
    sc = Scenario(w, oracle=full_oracle)
    full_plan = nk.nk_decode_workspace_bytes(sc.gpu.handle, w.B, w.T, w.Hq)
    assert (full_plan > SCRATCH_BYTES) == lowered, full_plan
    dev = "cuda"
    k, v = w.step_kv(0)
    q_cpu = w.step_q(0)
    q = q_cpu.to(dev)
    rows = torch.from_numpy(w.table_rows).to(dev)
    fr = torch.from_numpy(w.context + w.T).to(dev)
    if full_oracle:
        sc.orc.append(0, w.tables, w.table_rows, w.context, W.bf16_to_bits(k), W.bf16_to_bits(v))
    sc.gpu.append(0, sc.tables_d, rows, torch.from_numpy(w.context).to(dev), k.to(dev), v.to(dev))
    ref_out, ref_lse = sc.gpu.decode(0, q, sc.tables_d, rows, fr, w.scale)
    torch.cuda.synchronize()
    ref_out = ref_out.float().cpu().numpy().astype(np.float64)
    ref_lse = ref_lse.cpu().numpy().astype(np.float64)
    if full_oracle:
        orc_out, orc_lse = sc.oracle_decode(0, q_cpu, w.context + w.T)
        check = list(range(w.B))
    else:
        check = list(oracle_rows)
        pairs = [oracle_row(w, 0, b) for b in check]
        orc_out = np.stack([p[0] for p in pairs])
        orc_lse = np.stack([p[1] for p in pairs])
    for _ in range(2):               # two calls in a row share the static scratch
        out, lse = _noalloc(lib, sc, q, rows, fr, w)
        torch.cuda.synchronize()
        out, lse = out.cpu(), lse.cpu()
        compare_attention(out[check], lse[check], orc_out, orc_lse)   # the oracle
        # the workspace entry point: both outputs are bf16-rounded, so they
        # may differ by a full ulp (half from each side) beyond 2e-2
        compare_attention(out, lse, ref_out, ref_lse, ref_rounded=True)


def test_noalloc_plan_fits_the_scratch():
    """INT8-G64 decode batch (8 rows up to 4096 tokens, 16 q / 2 kv heads,
    D 256): the full split plan fits the array."""
    _run(W.int8_decode(num_layers=1))


def test_noalloc_k8v4_verify_fits_the_scratch():
    """K8V4 4-token verify (8 rows of 8192 tokens, 32 q / 4 kv heads, D 128)."""
    _run(W.k8v4_long(T=4, num_layers=1, S=8192), full_oracle=False, oracle_rows=[0, 5])


def test_noalloc_lowers_the_split_count():
    """INT8-G64, 4-token verify, 8 q heads per KV head, D 128: the warp-level
    kernel runs at least two CTAs per SM, and its full plan (a slot per CTA
    of a head's wave) needs more partials than the array holds, so the split
    budget per (row, KV head) is lowered, still above the 8 rows."""
    w = _workload("int8_g64", 2, 8, 128, 4, [4000, 3100, 2500, 4090, 1200, 3900, 64, 3000], seed=41)
    _run(w, lowered=True)


def test_noalloc_fewer_slots_than_rows():
    """FP8-row, 4-token verify over 16 KV heads with 8 q heads each, D 256:
    one split slot of all 8 rows x 16 heads x 32 query rows takes about
    4.2 MB, so the array holds 7 slots per (row, KV head), fewer than the 8
    rows.  Every row then runs as one split (written directly), one CTA per
    row: no row may be left out."""
    w = _workload("fp8_row", 16, 8, 256, 4, [700, 130, 450, 60, 1000, 333, 64, 900], seed=42)
    assert SCRATCH_BYTES // _split_bytes(w) < w.B
    _run(w, lowered=True)


def test_noalloc_lowers_the_pieces_of_the_tcgen05_kernel():
    """K8V4, 4-token verify over 8 KV heads with 8 q heads each, D 128, rows
    near 16k tokens: the transposed tcgen05 kernel plans 32 partial slots per
    (row, KV head), more than the array holds (31), so its piece budget is
    lowered to the slots that fit while pieces stay at least 64 pages long."""
    ctx = [16300, 16000, 15800, 16380, 15900, 16100, 16250, 16200]
    w = _workload("k8v4", 8, 8, 128, 4, ctx, seed=43, S=16384)
    assert 32 * _split_bytes(w) > SCRATCH_BYTES > 16 * _split_bytes(w)
    _run(w, full_oracle=False, oracle_rows=[3, 6], lowered=True)


def test_noalloc_rejects_calls_beyond_the_scratch():
    """8 rows x 256 KV heads x 16 query rows of head_dim 256 need more than
    the 32 MiB scratch even with one split per (row, head)."""
    lib = nk.load()
    H, G, T, D, B = 256, 8, 2, 256, 8
    assert B * H * G * T * (8 + 4 * D) + 256 > SCRATCH_BYTES
    pool = nk.Pool("int8_g64", 1, H, D, 64, B, B)
    dev = "cuda"
    q = torch.zeros((B, T, H * G, D), dtype=torch.bfloat16, device=dev)
    tables = torch.arange(B, dtype=torch.int32, device=dev).reshape(B, 1)
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    fr = torch.full((B,), 2, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    rc = lib.nk_paged_decode_attention_noalloc(
        q.data_ptr(), H * G, pool.handle, 0, tables.data_ptr(), rows.data_ptr(), fr.data_ptr(), B, T,
        ctypes.c_float(0.0625), out.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert rc == -7 and b"scratch" in lib.nk_last_error()
