"""The decode entry point that allocates nothing.

Callers that cannot allocate device memory (allocator callbacks, runtimes
whose memory budget is fixed at start-up, loops that must never block on
the driver's allocator) use nk_paged_decode_attention_noalloc, which keeps
the split-K partials in a static device array instead of a caller
workspace.  These tests call it through the C ABI and check that it returns
what nk_paged_decode_attention returns, within the parity tolerance, on two
calls in a row (the array keeps the previous call's contents), and that a
call too large for the array is rejected before any launch.

This file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_append_gb300 import nk
from paged_kv_cache_append_gb300 import workloads as W
from tests.scenario import Scenario

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20      # NK_NOALLOC_SCRATCH_BYTES in include/nk.h


def _close(out_a, lse_a, out_b, lse_b):
    a = out_a.float().cpu().numpy().astype(np.float64)
    b = out_b.float().cpu().numpy().astype(np.float64)
    excess = np.max(np.abs(a - b) - 2.0 ** -7 * np.abs(b))
    la, lb = lse_a.cpu().numpy(), lse_b.cpu().numpy()
    fin = np.isfinite(lb)
    assert np.array_equal(np.isfinite(la), fin)
    assert excess <= 2e-2, f"out differs by {excess} beyond one bf16 ulp"
    assert np.max(np.abs(la[fin] - lb[fin])) <= 1e-3


def _noalloc(lib, sc, q, rows, fr, w):
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], q.shape[1], q.shape[2]), float("nan"), device=q.device)
    rc = lib.nk_paged_decode_attention_noalloc(
        q.data_ptr(), w.Hq, sc.gpu.handle, 0, sc.tables_d.data_ptr(), rows.data_ptr(),
        fr.data_ptr(), q.shape[0], q.shape[1], ctypes.c_float(w.scale), out.data_ptr(),
        lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.nk_last_error().decode()
    return out, lse


@pytest.mark.parametrize("make", [lambda: W.int8_decode(num_layers=1),
                                  lambda: W.k8v4_long(T=4, num_layers=1, S=8192)],
                         ids=["int8_decode", "k8v4_verify"])
def test_noalloc_matches_workspace_entry_point(make):
    lib = nk.load()
    w = make()
    sc = Scenario(w, oracle=False)
    dev = "cuda"
    k, v = w.step_kv(0)
    q = w.step_q(0).to(dev)
    rows = torch.from_numpy(w.table_rows).to(dev)
    fr = torch.from_numpy(w.context + w.T).to(dev)
    sc.gpu.append(0, sc.tables_d, rows, torch.from_numpy(w.context).to(dev), k.to(dev), v.to(dev))
    ref_out, ref_lse = sc.gpu.decode(0, q, sc.tables_d, rows, fr, w.scale)
    for _ in range(2):               # two calls in a row share the static scratch
        out, lse = _noalloc(lib, sc, q, rows, fr, w)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)


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
