"""GPU parity of the host replica transfers ("Paged KV cache" page, host
replica section): pages packed in logical order by nk_pages_to_host equal the
oracle's packed pages byte for byte, for scattered pages (runs of one) and for
consecutive ones (one run); a replica restored by nk_pages_from_host into
other physical page groups reads back bit-identically through the remapped
table."""

import math

import numpy as np
import pytest
import torch

from paged_kv_cache_append_gb300 import nk
from paged_kv_cache_append_gb300 import workloads as W
from tests.scenario import Scenario

pytestmark = pytest.mark.gpu


def xfer_workload(profile, identity, seed):
    C, S, Hkv, G, D = 3, 700, 2, 8, 128
    L = -(-S // 64)
    rng = np.random.default_rng(seed)
    ids = np.arange(C * L, dtype=np.int32) if identity else rng.permutation(C * L).astype(np.int32)
    return W.Workload(f"xfer_{profile}", profile, 2, Hkv * G, Hkv, D, S, C, C * L, ids.reshape(C, L),
                      table_rows=np.arange(C, dtype=np.int32), context=np.array([100, 300, 50], np.int32),
                      T=1, scale=1 / math.sqrt(D), seed=seed + 100)


@pytest.mark.parametrize("profile", ["bf16", "int8_g64", "fp8_row", "nvfp4_g16", "k8v4"])
@pytest.mark.parametrize("identity", [False, True], ids=["scattered", "consecutive"])
@pytest.mark.parametrize("order", ["page_major", "head_major"])
def test_host_replica_round_trip(profile, identity, order):
    w = xfer_workload(profile, identity, seed=7 + identity)
    sc = Scenario(w, layers=(0, 1), order=order)
    src = w.tables[1, :5]                 # the 5 pages of row 1 (context 300)
    runs = nk.nk_page_runs(src)
    assert (len(runs) == 1) if identity else (len(runs) >= 2)
    pb = sc.gpu.host_page_bytes()
    assert pb == sc.orc.packed_page_bytes()
    host = torch.zeros((5, pb), dtype=torch.uint8).pin_memory()
    sc.gpu.pages_to_host(src, host)
    torch.cuda.synchronize()
    assert np.array_equal(host.numpy(), sc.orc.pack_pages(src))

    dst = w.tables[0, 2:7]                # pages row 0 (context 100) never reads
    sc.gpu.pages_from_host(dst, host)
    torch.cuda.synchronize()
    tables2 = w.tables.copy()
    tables2[1, :5] = dst
    dev = "cuda"
    tr = torch.tensor([1], dtype=torch.int32, device=dev)
    fr = torch.tensor([300], dtype=torch.int32, device=dev)
    for layer in (0, 1):
        q = w.step_q(layer)[1:2].to(dev)
        o1, l1 = sc.gpu.decode(layer, q, sc.tables_d, tr, fr, w.scale)
        o2, l2 = sc.gpu.decode(layer, q, torch.from_numpy(tables2).to(dev), tr, fr, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_transfer_rejects_out_of_range_page_ids():
    w = xfer_workload("int8_g64", False, seed=3)
    sc = Scenario(w, layers=(0,), oracle=False)
    host = torch.zeros((2, sc.gpu.host_page_bytes()), dtype=torch.uint8)
    with pytest.raises(nk.NkError):
        sc.gpu.pages_to_host([0, w.M], host)
    with pytest.raises(nk.NkError):
        sc.gpu.pages_from_host([-1, 0], host)
