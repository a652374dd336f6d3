"""Pins of oracle.attention: torch SDPA (library routine), brute force, closed forms."""

import math

import numpy as np
import pytest
import torch

from oracle import attention, formats as F
from oracle.store import PoolImage


def _sdpa_ref(q, K, V, n_keys_per_query, scale):
    """torch scaled_dot_product_attention in float64 with an explicit boolean
    mask; q [T, Hq, D], K/V [F, Hkv, D] (GQA expanded by repeat)."""
    T, Hq, D = q.shape
    G = Hq // K.shape[1]
    Kx = torch.from_numpy(np.repeat(K, G, axis=1)).permute(1, 0, 2)   # [Hq, F, D]
    Vx = torch.from_numpy(np.repeat(V, G, axis=1)).permute(1, 0, 2)
    qx = torch.from_numpy(q).permute(1, 0, 2)                          # [Hq, T, D]
    mask = torch.zeros(T, K.shape[0], dtype=torch.bool)
    for t, n in enumerate(n_keys_per_query):
        mask[t, :n] = True
    out = torch.nn.functional.scaled_dot_product_attention(qx, Kx, Vx, attn_mask=mask, scale=scale)
    s = torch.einsum("htd,hfd->htf", qx, Kx) * scale
    lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)
    return out.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("F_len,T", [(200, 1), (256, 1), (130, 4), (64, 4)])
def test_decode_matches_sdpa_bf16_identity(F_len, T):
    rng = np.random.default_rng(30)
    H, G, D, M = 2, 4, 64, 8
    k = F.f64_to_bf16_bits(rng.standard_normal((1, F_len, H, D)))
    v = F.f64_to_bf16_bits(rng.standard_normal((1, F_len, H, D)))
    pool = PoolImage("bf16", 1, H, D, M)
    table = np.arange(M, dtype=np.int32)[None]
    pool.append(0, table, np.array([0]), np.array([0]), k, v)
    K, V = pool.gather(0, table[0], F_len)
    q = F.bf16_bits_to_f64(F.f64_to_bf16_bits(rng.standard_normal((T, H * G, D))))
    scale = 1 / math.sqrt(D)
    out, lse = attention.decode(q, K, V, F_len, scale)
    ref_out, ref_lse = _sdpa_ref(q, K, V, [F_len - T + t + 1 for t in range(T)], scale)
    assert np.allclose(out, ref_out, atol=1e-12, rtol=1e-12)
    assert np.allclose(lse, ref_lse, atol=1e-12, rtol=1e-12)


def test_prefill_matches_sdpa():
    rng = np.random.default_rng(31)
    H, G, D = 2, 2, 32
    prefix, chunk, Tc = 77, 40, 48
    K = rng.standard_normal((prefix + chunk, H, D))
    V = rng.standard_normal((prefix + chunk, H, D))
    q = rng.standard_normal((Tc, H * G, D))
    out, lse = attention.prefill(q, K, V, prefix, chunk, 0.3)
    ref_out, ref_lse = _sdpa_ref(q[:chunk], K, V, [prefix + i + 1 for i in range(chunk)], 0.3)
    assert np.allclose(out[:chunk], ref_out, atol=1e-12)
    assert np.allclose(lse[:chunk], ref_lse, atol=1e-12)
    assert np.all(out[chunk:] == 0) and np.all(np.isneginf(lse[chunk:]))


def test_brute_force_loops():
    rng = np.random.default_rng(32)
    T, Hq, Hkv, D, Fl = 2, 4, 2, 3, 5
    q = rng.standard_normal((T, Hq, D))
    K = rng.standard_normal((Fl, Hkv, D))
    V = rng.standard_normal((Fl, Hkv, D))
    out, lse = attention.decode(q, K, V, Fl, 0.7)
    for t in range(T):
        for i in range(Hq):
            h = i * Hkv // Hq
            n = Fl - T + t + 1
            w = [math.exp(0.7 * sum(q[t, i, d] * K[j, h, d] for d in range(D))) for j in range(n)]
            z = sum(w)
            for d in range(D):
                assert abs(out[t, i, d] - sum(w[j] * V[j, h, d] for j in range(n)) / z) < 1e-12
            assert abs(lse[t, i] - math.log(z)) < 1e-12


def test_closed_form_zero_keys():
    rng = np.random.default_rng(33)
    Fl = 90
    K = np.zeros((Fl, 1, 16))
    V = rng.standard_normal((Fl, 1, 16))
    q = rng.standard_normal((1, 2, 16))
    out, lse = attention.decode(q, K, V, Fl, 0.25)
    assert np.allclose(lse, math.log(Fl), atol=1e-13)
    assert np.allclose(out[0, 0], V[:, 0].mean(axis=0), atol=1e-13)


def test_empty_key_set():
    out, lse = attention.decode(np.ones((1, 1, 4)), np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), 0, 1.0)
    assert np.all(out == 0) and np.isneginf(lse).all()


def test_verify_rows_equal_single_decodes():
    rng = np.random.default_rng(34)
    T, Fl = 4, 150
    q = rng.standard_normal((T, 8, 16))
    K = rng.standard_normal((Fl, 2, 16))
    V = rng.standard_normal((Fl, 2, 16))
    out, lse = attention.decode(q, K, V, Fl, 0.5)
    for t in range(T):
        o1, l1 = attention.decode(q[t:t + 1], K, V, Fl - T + t + 1, 0.5)
        assert np.allclose(out[t], o1[0], atol=1e-13) and np.allclose(lse[t], l1[0], atol=1e-13)


def test_mid_page_frontier_ignores_stale_tail():
    """Bytes past the frontier inside the last page (here NaN / max codes)
    are outside the valid domain and do not change the result."""
    rng = np.random.default_rng(35)
    H, D, M, Fl = 2, 64, 4, 200
    for profile in ("bf16", "int8_g64", "k8v4"):
        pool = PoolImage(profile, 1, H, D, M)
        table = np.array([[2, 0, 3, 1]], dtype=np.int32)
        k = F.f64_to_bf16_bits(rng.standard_normal((1, Fl, H, D)))
        pool.append(0, table, np.array([0]), np.array([0]), k, k)
        K0, V0 = pool.gather(0, table[0], Fl)
        q = rng.standard_normal((1, 4, D))
        ref = attention.decode(q, K0, V0, Fl, 0.125)
        g = int(table[0, Fl // 64])
        for pi, p in enumerate(pool.schema):
            for h in range(H):
                for o in range(Fl % 64, 64):
                    a = pool._row_slice(pi, o, h, g)
                    pool.planes[0][pi][a] = 0xFF
        K1, V1 = pool.gather(0, table[0], Fl)
        got = attention.decode(q, K1, V1, Fl, 0.125)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
