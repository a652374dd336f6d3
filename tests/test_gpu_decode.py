"""GPU parity of the paged append (bit-exact codes) and the paged decode /
verify attention (out max-abs 2e-2, LSE 1e-3) against the oracle, through the
C ABI."""

import math

import numpy as np
import pytest
import torch

from paged_kv_cache_append_gb300 import nk
from paged_kv_cache_append_gb300 import workloads as W
from tests.scenario import Scenario, compare_attention

pytestmark = pytest.mark.gpu


def small(profile, Hkv, G, D, S, C, T, seed, contexts=None, layers=1, outliers=True):
    rng = np.random.default_rng(seed)
    L = -(-S // 64)
    M = C * L
    tables = rng.permutation(M).astype(np.int32).reshape(C, L)
    ctx = np.asarray(contexts if contexts is not None else rng.integers(0, S - T + 1, C), np.int32)
    return W.Workload(f"small_{profile}", profile, layers, Hkv * G, Hkv, D, S, C, M, tables,
                      table_rows=np.arange(C, dtype=np.int32), context=ctx, T=T,
                      scale=1 / math.sqrt(D), seed=seed + 7000,
                      outlier_p=0.01 if outliers else 0.0, outlier_mul=20.0)


def run_and_check(w, layer=0, strict=False, fused=False, order="page_major"):
    sc = Scenario(w, layers=(layer,), order=order)
    q, out, lse, fr = sc.step(layer, fused=fused)
    bad = sc.planes_equal(layer)
    assert not bad, f"plane mismatch (plane, count, first index, gpu, oracle): {bad}"
    ref_out, ref_lse = sc.oracle_decode(layer, q, fr)
    return compare_attention(out, lse, ref_out, ref_lse, strict=strict)


def test_tiny_bf16_workload():
    """One sequence, frontier 200 (4 pages, 8 valid in the last), 8 q / 2 kv
    heads, D 128, pool of 8 pages in a seeded random order (plain 2e-2)."""
    run_and_check(W.tiny_bf16(), strict=True)


@pytest.mark.parametrize("profile", ["bf16", "int8_g64", "fp8_row", "nvfp4_g16", "k8v4"])
def test_no_outliers_plain_tolerance(profile):
    """N(0,1) data without outliers: |out| stays small, plain 2e-2 absolute."""
    w = small(profile, 2, 8, 128, 1000, 4, 1, seed=17, contexts=[0, 63, 500, 999], outliers=False)
    run_and_check(w, strict=True)


@pytest.mark.parametrize("profile", ["bf16", "int8_g64", "fp8_row", "nvfp4_g16", "k8v4"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G,T", [(8, 1), (4, 1), (1, 1), (2, 4), (8, 2)])
def test_small_shapes(profile, D, G, T):
    if D == 256 and G * T > 16:
        pytest.skip("head_dim 256 supports T*G <= 16")
    w = small(profile, 2, G, D, 300, 3, T, seed=D * 10 + G + T,
              contexts=[0, 137, 300 - T])
    run_and_check(w)


@pytest.mark.parametrize("profile", ["bf16", "int8_g64", "fp8_row", "nvfp4_g16", "k8v4"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G,T", [(8, 1), (2, 4), (8, 2)])
def test_fused_append_decode(profile, D, G, T):
    """nk_paged_append_decode_attention: the new tokens' codes are bit-exact
    (the whole layer's planes equal the oracle's) and the attention that reads
    them in the same launch matches the oracle."""
    if D == 256 and G * T > 16:
        pytest.skip("head_dim 256 supports T*G <= 16")
    w = small(profile, 2, G, D, 300, 3, T, seed=D * 10 + G + T + 1, contexts=[0, 137, 300 - T])
    run_and_check(w, fused=True)


@pytest.mark.parametrize("profile", ["int8_g64", "k8v4"])
def test_fused_new_tokens_straddle_pages_and_splits(profile):
    """T = 4 new tokens that straddle a page boundary (positions 126..129 and
    62..65), so that two CTAs of one row each encode part of them; plus rows
    long enough to be split."""
    w = small(profile, 4, 8, 128, 4096, 8, 4, seed=43,
              contexts=[126, 62, 0, 1020, 2046, 3000, 4092, 190])
    run_and_check(w, fused=True)


def test_fused_int8_decode_workload_one_layer():
    """The INT8-G64 decode workload's layer through the fused call."""
    run_and_check(W.int8_decode(num_layers=1), fused=True)


def test_row_without_keys_gets_zero_output():
    """A row whose frontier is 0 has no key: out = 0 and lse = -inf (the
    oracle's empty-set reading); the other rows are unaffected."""
    w = small("int8_g64", 2, 8, 128, 1024, 3, 1, seed=71, contexts=[0, 100, 700])
    sc = Scenario(w)
    dev = "cuda"
    q = w.step_q(0)
    tr = torch.from_numpy(w.table_rows).to(dev)
    fr_np = w.context.astype(np.int32)      # the filled context only; row 0 holds none
    fr = torch.from_numpy(fr_np).to(dev)
    out = torch.full((w.B, 1, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((w.B, 1, w.Hq), float("nan"), dtype=torch.float32, device=dev)
    sc.gpu.decode(0, q.to(dev), sc.tables_d, tr, fr, w.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    out, lse = out.cpu(), lse.cpu()
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ref_out, ref_lse = sc.oracle_decode(0, q, fr_np)
    compare_attention(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("profile", ["int8_g64", "k8v4"])
def test_verify_t4_gqa8(profile):
    """4-token verify (causal within the 4), 32 q / 4 kv heads, D 128."""
    w = small(profile, 4, 8, 128, 2048, 8, 4, seed=41, contexts=[4, 60, 61, 64, 500, 1000, 1500, 2044])
    run_and_check(w)


def test_int8_decode_workload_one_layer():
    """INT8-G64 decode batch of 8 rows, contexts uniform in [1, 4096], 16 q /
    2 kv heads, D 256, one layer of the 8, pool M = 512 shuffled."""
    run_and_check(W.int8_decode(num_layers=1))


def test_fp8_shared_prefix_with_cow_tail():
    """8 rows share a 1000-token prefix (15 full pages shared, 40 tail
    columns copied), then extend privately to mid-page frontiers."""
    w = W.fp8_shared(num_layers=2, C=8, S=4096, shared_len=1000)
    sc = Scenario(w, layers=(0, 1))
    for layer in (0, 1):
        q, out, lse, fr = sc.step(layer)
        assert not sc.planes_equal(layer)
        ref_out, ref_lse = sc.oracle_decode(layer, q, fr)
        compare_attention(out, lse, ref_out, ref_lse)


def test_stale_tail_bytes_are_not_read():
    """Bytes past the frontier inside each row's last page are set to 0xFF
    (NaN bf16 / max codes / NaN scales) on the GPU only; the results must
    stay finite and equal to the oracle's."""
    for profile in ("bf16", "int8_g64", "k8v4"):
        w = small(profile, 2, 8, 128, 1024, 4, 1, seed=51, contexts=[10, 200, 333, 700])
        sc = Scenario(w)
        k, v = w.step_kv(0)
        dev = "cuda"
        tr = torch.from_numpy(w.table_rows).to(dev)
        fr = torch.from_numpy(w.context + 1).to(dev)
        sc.gpu.append(0, sc.tables_d, tr, torch.from_numpy(w.context).to(dev), k.to(dev), v.to(dev))
        from paged_kv_cache_append_gb300.workloads import bf16_to_bits
        sc.orc.append(0, w.tables, w.table_rows, w.context, bf16_to_bits(k), bf16_to_bits(v))
        for b in range(w.B):
            F = int(w.context[b]) + 1
            g = int(w.tables[b, F // 64])
            for i, plane in enumerate(sc.gpu.planes[0]):
                rb = sc.gpu.row_bytes[i]
                for h in range(w.Hkv):
                    base = ((g * w.Hkv + h) * 64) * rb
                    plane[base + (F % 64) * rb: base + 64 * rb] = 0xFF
        q = w.step_q(0)
        out, lse = sc.gpu.decode(0, q.to(dev), sc.tables_d, tr, fr, w.scale)
        ref_out, ref_lse = sc.oracle_decode(0, q, w.context + 1)
        compare_attention(out.cpu(), lse.cpu(), ref_out, ref_lse)


def test_physical_order_and_row_selection_do_not_change_results():
    """Same logical content under two random physical-page permutations gives
    bit-identical results; permuting table_rows permutes the outputs."""
    base = small("fp8_row", 2, 8, 128, 2048, 6, 1, seed=61, contexts=[5, 64, 65, 700, 1500, 2047])
    outs = []
    for seed in (1, 2):
        w = small("fp8_row", 2, 8, 128, 2048, 6, 1, seed=61, contexts=base.context)
        w.tables = np.random.default_rng(seed).permutation(w.M).astype(np.int32).reshape(w.C, w.L)
        sc = Scenario(w, oracle=False)
        _, out, lse, _ = sc.step(0)
        outs.append((out, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    # compact-row order is independent of table-row order
    w = small("fp8_row", 2, 8, 128, 2048, 6, 1, seed=61, contexts=base.context)
    sc = Scenario(w, oracle=False)
    k, v = w.step_kv(0)
    q = w.step_q(0)
    dev = "cuda"
    sc.gpu.append(0, sc.tables_d, torch.arange(6, dtype=torch.int32, device=dev),
                  torch.from_numpy(w.context).to(dev), k.to(dev), v.to(dev))
    perm = np.array([3, 0, 5, 1, 4, 2])
    o1, l1 = sc.gpu.decode(0, q.to(dev), sc.tables_d, torch.arange(6, dtype=torch.int32, device=dev),
                           torch.from_numpy(w.context + 1).to(dev), w.scale)
    o2, l2 = sc.gpu.decode(0, q[perm].contiguous().to(dev), sc.tables_d,
                           torch.from_numpy(perm.astype(np.int32)).to(dev),
                           torch.from_numpy((w.context + 1)[perm]).to(dev), w.scale)
    assert torch.equal(o1[perm], o2) and torch.equal(l1[perm], l2)


def test_bounds_mode_flags_bad_page_ids():
    w = small("int8_g64", 2, 8, 64, 512, 2, 1, seed=71, contexts=[100, 300])
    sc = Scenario(w, oracle=False, check_bounds=True)
    nk.nk_status_read(clear=True)
    bad = sc.tables_d.clone()
    bad[1, 2] = w.M + 5                     # a page id outside [0, M)
    q = w.step_q(0).cuda()
    sc.gpu.decode(0, q, bad, torch.arange(2, dtype=torch.int32, device="cuda"),
                  torch.tensor([101, 301], dtype=torch.int32, device="cuda"), w.scale)
    assert nk.nk_status_read(clear=True) & nk.STATUS_PAGE_RANGE
    fr = torch.tensor([101, 10_000], dtype=torch.int32, device="cuda")   # past L * 64
    sc.gpu.decode(0, q, sc.tables_d, torch.arange(2, dtype=torch.int32, device="cuda"), fr, w.scale)
    assert nk.nk_status_read(clear=True) & nk.STATUS_FRONTIER
    assert nk.nk_status_read(clear=True) == 0


def test_argument_errors_launch_nothing():
    w = small("bf16", 2, 4, 64, 256, 2, 1, seed=81, contexts=[10, 20])
    sc = Scenario(w, oracle=False)
    q = w.step_q(0).cuda()
    tr = torch.arange(2, dtype=torch.int32, device="cuda")
    fr = torch.tensor([11, 21], dtype=torch.int32, device="cuda")
    with pytest.raises(nk.NkError) as e:
        sc.gpu.decode(0, q, sc.tables_d, tr, fr, w.scale,
                      workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == -7
    with pytest.raises(nk.NkError) as e:
        sc.gpu.decode(0, q[:, :, :7].contiguous(), sc.tables_d, tr, fr, w.scale)
    assert e.value.code == -2
    with pytest.raises(nk.NkError) as e:
        sc.gpu.decode(5, q, sc.tables_d, tr, fr, w.scale)
    assert e.value.code == -2


def test_negative_softmax_scale():
    """Decode with a negative softmax scale (the score order reverses)."""
    import dataclasses
    w = small("fp8_row", 2, 8, 128, 700, 3, 1, seed=81, contexts=[5, 300, 699])
    run_and_check(dataclasses.replace(w, scale=-w.scale))


@pytest.mark.parametrize("profile", ["int8_g64", "k8v4", "bf16"])
def test_rejected_speculative_tail_is_never_read_and_is_overwritten(profile):
    """Rollback of a speculative round.  A 4-token verify (fused call) writes
    and attends 4 provisional tokens; only the first is accepted, so the
    committed frontier is context + 1 and the 3 rejected tokens stay in the
    page.  Their bytes are then poisoned (0xFF) on the GPU only.  The next
    decode appends one token at the committed frontier and attends up to it:
    the result matches the oracle (which never holds the poison), and the
    codes of the rewritten position are bit-exact."""
    import dataclasses
    w4 = small(profile, 2, 8, 128, 1024, 3, 4, seed=91, contexts=[60, 126, 500])
    sc = Scenario(w4)
    q, out, lse, fr = sc.step(0, fused=True)
    ref_out, ref_lse = sc.oracle_decode(0, q, fr)
    compare_attention(out, lse, ref_out, ref_lse)
    committed = (w4.context + 1).astype(np.int32)

    def rows_at(pos_of_b):
        """(gpu, oracle) bytes of every plane at one position per row."""
        got, want = [], []
        for b in range(w4.B):
            pos = int(pos_of_b[b])
            g = int(w4.tables[w4.table_rows[b], pos // 64])
            for i, plane in enumerate(sc.gpu.planes[0]):
                rb = sc.gpu.row_bytes[i]
                for h in range(w4.Hkv):
                    off = ((g * w4.Hkv + h) * 64 + pos % 64) * rb
                    got.append(plane[off:off + rb].cpu().numpy())
                    want.append(sc.orc.planes[0][i][off:off + rb])
        return np.concatenate(got), np.concatenate(want)

    for b in range(w4.B):                       # poison the rejected tail on the GPU
        for pos in range(int(committed[b]), int(fr[b])):
            g = int(w4.tables[w4.table_rows[b], pos // 64])
            for i, plane in enumerate(sc.gpu.planes[0]):
                rb = sc.gpu.row_bytes[i]
                for h in range(w4.Hkv):
                    off = ((g * w4.Hkv + h) * 64 + pos % 64) * rb
                    plane[off:off + rb] = 0xFF
    sc.w = dataclasses.replace(w4, T=1, context=committed, seed=w4.seed + 1)
    q1, out1, lse1, fr1 = sc.step(0, fused=True)
    assert np.array_equal(fr1, committed + 1)
    ref_out1, ref_lse1 = sc.oracle_decode(0, q1, fr1)
    compare_attention(out1, lse1, ref_out1, ref_lse1)
    got, want = rows_at(committed)
    assert np.array_equal(got, want), "rewritten position differs from the oracle"


@pytest.mark.parametrize("profile", ["bf16", "int8_g64", "fp8_row", "nvfp4_g16", "k8v4"])
@pytest.mark.parametrize("D,G,T", [(128, 8, 1), (256, 8, 1), (128, 2, 4)])
@pytest.mark.parametrize("fused", [False, True], ids=["append_then_decode", "fused"])
def test_head_major_plane_order(profile, D, G, T, fused):
    """Pools in the head-major order [X, P, N, H] of the draft pool: the
    append writes, and the decode reads, the same logical content as the
    oracle's head-major image (planes bit-exact, attention within tolerance)."""
    w = small(profile, 2, G, D, 400, 3, T, seed=D + G + T + 300, contexts=[0, 190, 400 - T])
    run_and_check(w, fused=fused, order="head_major")


def test_head_major_shared_prefix_with_cow_tail():
    """Fork with a partial-tail copy (nk_page_copy_columns) in a head-major
    pool: the per-head column runs sit M pages apart."""
    w = W.fp8_shared(num_layers=1, C=4, S=2048, shared_len=1000)
    sc = Scenario(w, layers=(0,), order="head_major")
    q, out, lse, fr = sc.step(0, fused=True)
    assert not sc.planes_equal(0)
    ref_out, ref_lse = sc.oracle_decode(0, q, fr)
    compare_attention(out, lse, ref_out, ref_lse)


# ---- 17..32 query rows per KV head over FP8-row / NVFP4-G16 / K8V4 pages --------
# These shapes run the tcgen05 decode kernel (Q and the accumulators in tensor
# memory); the same split plan and merge as the warp-level kernel.

@pytest.mark.parametrize("profile", ["fp8_row", "nvfp4_g16", "k8v4"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G,T", [(8, 4), (6, 3), (32, 1), (16, 2)])
@pytest.mark.parametrize("fused", [False, True], ids=["append_then_decode", "fused"])
def test_wide_query_groups(profile, D, G, T, fused):
    """T * G in 17..32 (18 leaves a ragged last 8-row group): a row with a
    frontier inside its first page, one just past a page edge, and one long
    enough to be split."""
    Hkv = 1 if G >= 16 else 2
    w = small(profile, Hkv, G, D, 3000, 3, T, seed=D * 7 + G * 3 + T + (1 if fused else 0),
              contexts=[0, 62, 3000 - T])
    run_and_check(w, fused=fused)


@pytest.mark.parametrize("profile", ["fp8_row", "nvfp4_g16", "k8v4"])
def test_wide_query_groups_stale_tail_and_negative_scale(profile):
    """Bytes past each frontier poisoned with 0xFF on the GPU (NaN codes and
    scales), and a negative softmax scale, at T * G = 32."""
    import dataclasses
    w = small(profile, 2, 8, 128, 1024, 4, 4, seed=61, contexts=[10, 200, 333, 700])
    w = dataclasses.replace(w, scale=-w.scale)
    sc = Scenario(w)
    k, v = w.step_kv(0)
    dev = "cuda"
    tr = torch.from_numpy(w.table_rows).to(dev)
    fr = torch.from_numpy(w.context + 4).to(dev)
    sc.gpu.append(0, sc.tables_d, tr, torch.from_numpy(w.context).to(dev), k.to(dev), v.to(dev))
    from paged_kv_cache_append_gb300.workloads import bf16_to_bits
    sc.orc.append(0, w.tables, w.table_rows, w.context, bf16_to_bits(k), bf16_to_bits(v))
    for b in range(w.B):
        F = int(w.context[b]) + 4
        g = int(w.tables[b, F // 64])
        for i, plane in enumerate(sc.gpu.planes[0]):
            rb = sc.gpu.row_bytes[i]
            for h in range(w.Hkv):
                base = ((g * w.Hkv + h) * 64) * rb
                plane[base + (F % 64) * rb: base + 64 * rb] = 0xFF
    q = w.step_q(0)
    out, lse = sc.gpu.decode(0, q.to(dev), sc.tables_d, tr, fr, w.scale)
    ref_out, ref_lse = sc.oracle_decode(0, q, w.context + 4)
    compare_attention(out.cpu(), lse.cpu(), ref_out, ref_lse)


@pytest.mark.parametrize("profile", ["fp8_row", "k8v4"])
@pytest.mark.parametrize("fused", [False, True], ids=["append_then_decode", "fused"])
def test_wide_query_groups_head_major(profile, fused):
    w = small(profile, 2, 8, 256, 700, 3, 4, seed=307, contexts=[0, 190, 696])
    run_and_check(w, fused=fused, order="head_major")


def test_wide_query_groups_at_head_dim_256_need_exact_f16_codes():
    """T * G > 16 at head_dim 256 is served by the tcgen05 kernel only; the
    BF16 and INT8-G64 profiles reject it before launching anything."""
    for profile in ("bf16", "int8_g64"):
        w = small(profile, 2, 8, 256, 300, 2, 4, seed=5, contexts=[10, 20])
        sc = Scenario(w, oracle=False)
        dev = "cuda"
        with pytest.raises(nk.NkError) as e:
            sc.gpu.decode(0, w.step_q(0).to(dev), sc.tables_d, torch.from_numpy(w.table_rows).to(dev),
                          torch.from_numpy(w.context + 4).to(dev), w.scale)
        assert e.value.code == -4   # NK_ERR_UNSUPPORTED


# ---- many KV heads: a per-head split budget below the number of rows ------------
@pytest.mark.parametrize("profile,Hkv,G,D,T", [
    ("fp8_row", 24, 8, 256, 4),     # tcgen05 quadrant kernel, one CTA per SM: 152 / 24 = 6 < 8 rows
    ("k8v4", 40, 8, 128, 4),        # transposed tcgen05 kernel (pieces): 152 / 40 = 3 < 8 rows
    ("int8_g64", 64, 8, 256, 1),    # warp-level kernel at D 256: (152 x CTAs per SM) / 64 < 8 rows
], ids=["quadrant", "pieces", "warp_level"])
@pytest.mark.parametrize("fused", [False, True], ids=["append_then_decode", "fused"])
def test_many_kv_heads_still_cover_every_row(profile, Hkv, G, D, T, fused):
    """With so many KV heads that the SMs give each head fewer CTAs than the
    batch has rows, every row still runs (one split each) and matches the
    oracle; no row is left unwritten."""
    w = small(profile, Hkv, G, D, 256, 8, T, seed=Hkv + D + T,
              contexts=[0, 60, 100, 127, 190, 200, 250 - T, 63])
    run_and_check(w, fused=fused)
