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


# ------------------------------------------------ speculative page geometry

def test_pages_needed_counts_the_touched_pages():
    """ceil(max(committed, provisional) / P) equals the number of distinct
    pages that positions [0, max) touch (brute force)."""
    for c in range(0, 300, 7):
        for p_ in range(0, 300, 11):
            touched = len({pos >> 6 for pos in range(max(c, p_))})
            assert layout.pages_needed(c, p_) == touched


def test_mtp_pool_covers_the_worst_provisional_lead():
    """The MTP pool's extra pages per row equal the largest number of pages a
    lead of K - 1 provisional tokens can add beyond Main's membership, over
    every committed frontier offset (brute force over a few pages)."""
    for K in range(1, 200):
        worst = max(layout.pages_needed(f, f + K - 1) - layout.pages_needed(f, f) for f in range(0, 4 * 64))
        for M, C in [(1, 1), (512, 8), (16384, 8)]:
            assert layout.mtp_pages(M, C, K) == M + C * worst
    assert layout.mtp_pages(512, 8, 1) == 512            # no draft lead, no extra page
    assert layout.mtp_pages(512, 8, 65) == 512 + 8        # a 64-token lead fits one page
    assert layout.mtp_pages(512, 8, 66) == 512 + 16


# ------------------------------------------------------------ host replica

def _filled_image(profile, layers=2, H=2, D=64, M=6, seed=5):
    from oracle.store import PoolImage
    rng = np.random.default_rng(seed)
    img = PoolImage(profile, layers, H, D, M)
    for layer in range(layers):
        for pi in range(len(img.schema)):
            img.planes[layer][pi][:] = rng.integers(0, 256, img.planes[layer][pi].size, dtype=np.uint8)
    return img


@pytest.mark.parametrize("profile", ["bf16", "int8_g64", "k8v4"])
def test_packed_page_is_the_page_major_slice_of_every_plane(profile):
    """In the page-major order one page group is one contiguous byte range of
    each plane, so a packed page is those ranges concatenated (layer-major,
    then plane order) -- checked by plain slicing, not by row addressing."""
    img = _filled_image(profile)
    ids = [4, 0, 5, 2]
    packed = img.pack_pages(ids)
    for i, g in enumerate(ids):
        expect = []
        for layer in range(img.num_layers):
            for pi, p in enumerate(img.schema):
                n = p.row_bytes * 64 * img.H
                expect.append(img.planes[layer][pi][g * n:(g + 1) * n])
        assert np.array_equal(packed[i], np.concatenate(expect))


def test_packed_page_size_matches_the_page_byte_table():
    """Packed page bytes = layers x PageBytes (sum over planes of bytes per
    token-head x 64 x H), the page's PageBytes definition."""
    from oracle.store import PoolImage
    for profile in layout.PROFILES:
        img = PoolImage(profile, 3, 2, 256, 4)
        assert img.packed_page_bytes() == layout.page_bytes(profile, 256, 2, 3)


def test_unpack_into_other_pages_reads_the_same_logical_content():
    """A replica restored into different physical page groups, with the
    table row remapped, gathers to the same logical values."""
    from oracle.store import PoolImage
    img = _filled_image("fp8_row", layers=1, H=2, D=64, M=8)
    src = np.array([3, 1, 6], np.int32)
    dst = np.array([0, 7, 2], np.int32)
    img.unpack_pages(dst, img.pack_pages(src))
    r1, r2 = img.read_rows(0, src, 3 * 64), img.read_rows(0, dst, 3 * 64)
    assert all(np.array_equal(r1[k], r2[k]) for k in r1)
