"""GPU parity at the full per-layer size of the large decode workloads, one
layer, on sampled rows: the FP8-row shared-prefix batch (8 rows of ~32.7k
tokens sharing 16384 tokens of pages), the K8V4 long-context batch (8 rows of
131072 tokens) and its 4-token verify.  The GPU runs the fused append + decode
call over the whole batch (full split plan and merge); the oracle encodes,
decodes and attends the sampled rows from the same host-drawn inputs."""

import numpy as np
import pytest
import torch

import bench
from oracle import attention as OA
from oracle import codec as OC
from oracle import formats as OF
from paged_kv_cache_append_gb300.workloads import bf16_to_bits
from tests.scenario import compare_attention

pytestmark = pytest.mark.gpu


def oracle_row(w, layer, b):
    """(out [T, Hq, D], lse [T, Hq]) of decode row b, from host inputs."""
    r = int(w.table_rows[b])
    n = int(w.context[b])
    sh = w.shared_len
    kc, vc = w.context_kv(layer, r, n)
    if sh and r != 0:                       # the shared prefix holds row 0's values
        k0, v0 = w.context_kv(layer, 0, int(w.context[0]))
        kc = torch.cat([k0[:sh], kc[sh:]])
        vc = torch.cat([v0[:sh], vc[sh:]])
    ks, vs = w.step_kv(layer)
    kb = np.concatenate([bf16_to_bits(kc), bf16_to_bits(ks[b])], axis=0)
    vb = np.concatenate([bf16_to_bits(vc), bf16_to_bits(vs[b])], axis=0)
    K, V = OC.decode_kv(w.profile, OC.encode_kv(w.profile, kb, vb))
    q = OF.bf16_bits_to_f64(bf16_to_bits(w.step_q(layer)[b]))
    return OA.decode(q, K, V, n + w.T, w.scale)


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
