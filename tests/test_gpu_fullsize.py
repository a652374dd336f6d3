"""GPU parity at the full per-layer size of the large decode workloads, one
layer, on sampled rows: the FP8-row shared-prefix batch (8 rows of ~32.7k
tokens sharing 16384 tokens of pages), the K8V4 long-context batch (8 rows of
131072 tokens) and its 4-token verify.  The GPU runs the fused append + decode
call over the whole batch (full split plan and merge); the oracle encodes,
decodes and attends the sampled rows from the same host-drawn inputs."""

import pytest
import torch

import bench
from tests.scenario import compare_attention, oracle_row

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,rows", [("fp8_shared", [0, 5]), ("k8v4_long", [2, 7]), ("k8v4_verify", [4])])
def test_full_size_workload_sampled_rows(name, rows):
    w = bench.make_workload(name, layers=1)
    bn = bench.Bench(w, "cuda", host_values=True)
    bn.attend(0)
    torch.cuda.synchronize()
    out, lse = bn.out[0].cpu(), bn.lse[0].cpu()
    for b in rows:
        ref_o, ref_l = oracle_row(w, 0, b)
        compare_attention(out[b], lse[b], ref_o, ref_l)
