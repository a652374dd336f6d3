"""Pins of oracle.layout and oracle.store: closed forms, hand-computed
addresses, the Fork worked example, permutation invariance, COW."""

import os

import numpy as np
import pytest

from oracle import formats as F, layout
from oracle.store import PoolImage

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("S,C,lo,hi", [
    (512, 1, 8, 8), (4096, 8, 64, 512), (32768, 8, 512, 4096), (131072, 8, 2048, 16384),
    (1, 8, 8, 8), (63, 3, 3, 3), (65, 2, 2, 4), (64, 1, 1, 1)])
def test_capacity_bounds_closed_form(S, C, lo, hi):
    # L = ceil(S/64); M_min = max(L, C); M_max = C * L
    assert layout.m_bounds(S, C) == (lo, hi)


def test_explicit_capacity_policy():
    assert layout.explicit_capacity(4096 * 8, 4096, 8) == 512
    assert layout.explicit_capacity(4096, 4096, 8) == 64
    assert layout.explicit_capacity(4097, 4096, 8) == 65       # page rounding
    with pytest.raises(ValueError):
        layout.explicit_capacity(4000, 4096, 8)                # K_main < S
    with pytest.raises(ValueError):
        layout.explicit_capacity(4096 * 8 + 1, 4096, 8)        # M > M_max
    with pytest.raises(ValueError):
        layout.explicit_capacity(100, 64, 4)                   # M = 2 < C = 4


def test_addresses_by_hand():
    k = layout.plane_schema("int8_g64", 256)[0]        # X = 256, 1 byte
    # page-major [X, P, H, N]: nb = (1, 256, 64*256, 2*64*256)
    assert layout.strides(k, 2, 4) == (1, 256, 16384, 32768)
    assert layout.address(k, 2, 4, d=5, o=3, h=1, g=2) == 5 + 3 * 256 + 16384 + 2 * 32768
    # head-major [X, P, N, H]: nb2 = 64*256, nb3 = N*64*256
    assert layout.address(k, 2, 4, 5, 3, 1, 2, "head_major") == 5 + 768 + 2 * 16384 + 65536
    ks = layout.plane_schema("int8_g64", 256)[2]       # X = 4, 2 bytes
    assert layout.strides(ks, 2, 4) == (2, 8, 512, 1024)
    v = layout.plane_schema("k8v4", 128)[1]            # packed NVFP4, X = 64
    assert layout.address(v, 4, 16, d=10, o=63, h=3, g=1) == 10 + 63 * 64 + 3 * 4096 + 16384


def test_translation():
    row = np.array([5, 3, 7, 1, 0, 2, 6, 4], dtype=np.int32)
    assert layout.translate(0, row) == (5, 0)
    assert layout.translate(63, row) == (5, 63)
    assert layout.translate(64, row) == (3, 0)
    assert layout.translate(199, row) == (1, 7)      # frontier 200: 4th page, 8 valid
    assert layout.translate(511, row) == (4, 63)


def test_fork_worked_example():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "fork_cow_example.txt"))
            if l.strip() and not l.startswith("#")]
    for Pp, Fr, full, tail, not_rounded in rows:
        assert int(Pp) == layout.P
        assert layout.fork_split(int(Fr)) == (int(full), int(tail))
        assert int(full) * layout.P + int(tail) == int(Fr) != int(not_rounded)


def _bits(rng, shape):
    return F.f64_to_bf16_bits(rng.standard_normal(shape))


@pytest.mark.parametrize("profile", layout.PROFILES)
def test_pool_round_trip_and_permutation_invariance(profile):
    rng = np.random.default_rng(20)
    H, D, M, T = 2, 64, 6, 300
    k = _bits(rng, (1, T, H, D))
    v = _bits(rng, (1, T, H, D))
    ident = PoolImage(profile, 1, H, D, M)
    perm = PoolImage(profile, 1, H, D, M)
    t_id = np.arange(M, dtype=np.int32)[None, :5]
    t_pm = rng.permutation(M).astype(np.int32)[None, :5]
    for pool, tab in ((ident, t_id), (perm, t_pm)):
        pool.append(0, tab, np.array([0]), np.array([0]), k, v)
    K1, V1 = ident.gather(0, t_id[0], T)
    K2, V2 = perm.gather(0, t_pm[0], T)
    assert np.array_equal(K1, K2) and np.array_equal(V1, V2)
    # BF16 stores bits unchanged; other profiles reproduce the codec's values
    if profile == "bf16":
        assert np.array_equal(K1, F.bf16_bits_to_f64(k[0]))
    # plane bytes are at the page-major addresses of the translated positions
    p0 = perm.schema[0]
    g, o = layout.translate(130, t_pm[0])
    a = layout.address(p0, H, M, 0, o, 1, g)
    assert np.array_equal(perm.planes[0][0][a:a + p0.row_bytes],
                          ident.planes[0][0][layout.address(p0, H, M, 0, 130 % 64, 1, 130 // 64):][:p0.row_bytes])


def test_plane_sizes_sum_to_page_bytes():
    for prof in layout.PROFILES:
        pool = PoolImage(prof, 2, 2, 128, 3)
        tot = sum(a.size for layer in pool.planes for a in layer)
        assert tot == layout.page_bytes(prof, 128, 2, num_layers=2) * 3


def test_shared_prefix_fork_reads_identically():
    """Fork at F = 1000: 15 shared full pages, a private tail page with the 40
    committed columns; forked rows read the source prefix bit-for-bit, later
    appends only write private pages, shared pages stay unchanged."""
    rng = np.random.default_rng(21)
    H, D, Fk, M, C = 2, 64, 1000, 64, 3
    pool = PoolImage("int8_g64", 2, H, D, M)
    src = np.arange(16, dtype=np.int32)                  # pages 0..15 of the source
    tables = np.zeros((C + 1, 20), dtype=np.int32)
    tables[0, :16] = src
    k = _bits(rng, (1, Fk, H, D))
    v = _bits(rng, (1, Fk, H, D))
    for layer in range(2):
        pool.append(layer, tables, np.array([0]), np.array([0]), k, v)
    full, tail = layout.fork_split(Fk)
    nxt = 16
    for r in range(1, C + 1):
        tables[r, :full] = src[:full]                     # shared immutable pages
        tables[r, full:20] = np.arange(nxt, nxt + 20 - full)
        pool.copy_columns(int(src[full]), int(tables[r, full]), tail)
        nxt += 20 - full
    snap = [[a.copy() for a in layer] for layer in pool.planes]
    ref = [pool.gather(layer, tables[0], Fk) for layer in range(2)]
    for r in range(1, C + 1):
        for layer in range(2):
            Kr, Vr = pool.gather(layer, tables[r], Fk)
            assert np.array_equal(Kr, ref[layer][0]) and np.array_equal(Vr, ref[layer][1])
    # private appends after the fork
    kk = _bits(rng, (C, 100, H, D))
    vv = _bits(rng, (C, 100, H, D))
    for layer in range(2):
        pool.append(layer, tables, np.arange(1, C + 1), np.full(C, Fk), kk, vv)
    for layer in range(2):
        for pi, p in enumerate(pool.schema):
            for g in src[:full]:
                lo = layout.address(p, H, M, 0, 0, 0, int(g))
                hi = lo + H * 64 * p.row_bytes
                assert np.array_equal(pool.planes[layer][pi][lo:hi], snap[layer][pi][lo:hi])
    # each row now reads its own suffix
    for r in range(1, C + 1):
        Kr, _ = pool.gather(1, tables[r], Fk + 100)
        Kexp, _ = PoolImage_gather_direct("int8_g64", kk[r - 1])
        assert np.array_equal(Kr[Fk:], Kexp)


def PoolImage_gather_direct(profile, bits):
    from oracle import codec
    return codec.decode_kv(profile, codec.encode_kv(profile, bits, bits))
