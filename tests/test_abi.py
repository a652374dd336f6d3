"""CPU checks of the C-ABI library: it loads, exports every symbol that
include/nk.h declares, and its host-only calls agree with the oracle's
geometry.  No kernel is launched here."""

import ctypes
import os
import re

import pytest

from oracle import layout
from paged_kv_cache_append_gb300 import build, nk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(nk.LIB_PATH):
        build.build()
    return nk.load()


def test_exports_every_declared_symbol(lib):
    header = open(os.path.join(ROOT, "include", "nk.h")).read()
    declared = set(re.findall(r"^\s*(?:int|const char\*)\s+(nk_\w+)\s*\(", header, re.M))
    assert declared == set(nk.SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_version(lib):
    assert nk.nk_version() >= 100


@pytest.mark.parametrize("profile", layout.PROFILES)
@pytest.mark.parametrize("D", [64, 128, 256])
def test_plane_bytes_match_oracle_layout(lib, profile, D):
    H, M = 3, 17
    desc = nk.make_desc(profile, 2, H, D, 1024, 2)
    n, sizes, rows = nk.nk_pool_plane_bytes(desc, M)
    schema = layout.plane_schema(profile, D)
    assert n == len(schema)
    assert rows == [p.row_bytes for p in schema]
    assert sizes == [layout.plane_bytes(p, H, M) for p in schema]


@pytest.mark.parametrize("S,C", [(512, 1), (4096, 8), (32768, 8), (131072, 8), (1, 8), (65, 2)])
def test_capacity_bounds_match_oracle(lib, S, C):
    desc = nk.make_desc("int8_g64", 1, 2, 128, S, C)
    assert nk.nk_pool_capacity_bounds(desc) == layout.m_bounds(S, C)


def test_pool_create_rejects_m_outside_bounds(lib):
    desc = nk.make_desc("fp8_row", 1, 2, 128, 4096, 8)
    lo, hi = nk.nk_pool_capacity_bounds(desc)
    for M in (lo - 1, hi + 1):
        with pytest.raises(nk.NkError) as e:
            nk.nk_pool_create(desc, M, [16] * 4)
        assert e.value.code == -3 and "outside" in str(e.value)


def test_host_argument_errors(lib):
    with pytest.raises(nk.NkError) as e:
        nk.nk_pool_plane_bytes(nk.make_desc("bf16", 1, 2, 96, 64, 1), 4)
    assert e.value.code == -4                      # head_dim 96 not built
    with pytest.raises(nk.NkError) as e:
        nk.nk_pool_plane_bytes(nk.make_desc(9, 1, 2, 64, 64, 1), 4)
    assert e.value.code == -1                      # unknown profile
    with pytest.raises(nk.NkError) as e:
        nk.nk_pool_capacity_bounds(nk.make_desc("bf16", 1, 2, 64, 64, 9))
    assert e.value.code == -2                      # C > 8
    desc = nk.make_desc("bf16", 1, 2, 64, 4096, 2)
    lo, _ = nk.nk_pool_capacity_bounds(desc)
    with pytest.raises(nk.NkError) as e:
        nk.nk_pool_create(desc, lo, [0, 0])
    assert e.value.code == -1                      # null plane pointer
    with pytest.raises(nk.NkError) as e:
        nk.nk_pool_create(desc, lo, [8, 16])
    assert e.value.code == -5                      # misaligned plane pointer
    # calls on a NULL pool fail before any launch
    assert lib.nk_paged_kv_append(None, 0, None, None, None, None, None, None, 1, 1, None) == -1
    assert lib.nk_paged_decode_attention(None, 8, None, 0, None, None, None, 1, 1, 1.0,
                                         None, None, None, 0, None) == -1
    assert lib.nk_page_copy_columns(None, 0, 1, 4, None) == -1
    assert lib.nk_last_error()


def test_speculative_page_geometry_matches_oracle():
    """nk_pool_mtp_pages and nk_pages_needed are host arithmetic: checked
    against the oracle without a GPU, including their range errors."""
    from oracle import layout
    for M, Cr, K in [(1, 1, 1), (512, 8, 4), (512, 8, 65), (16384, 8, 129), (4096, 2, 200)]:
        assert nk.nk_pool_mtp_pages(M, Cr, K) == layout.mtp_pages(M, Cr, K)
    for c, p_ in [(0, 0), (1, 0), (64, 64), (65, 3), (1000, 1004), (4092, 4096)]:
        assert nk.nk_pages_needed(c, p_) == layout.pages_needed(c, p_)
    with pytest.raises(nk.NkError):
        nk.nk_pool_mtp_pages(512, 8, 0)
    with pytest.raises(nk.NkError):
        nk.nk_pages_needed(-1, 5)


def test_page_runs_merge_consecutive_physical_ids():
    """nk_page_runs (host code): runs of ids that increase by one in logical
    order, against a plain loop."""
    import numpy as np
    rng = np.random.default_rng(3)
    cases = [[], [7], [3, 4, 5, 9, 10, 2], list(range(20)), [5, 4, 3], rng.permutation(40).tolist(),
             [0, 1, 1, 2]]
    for ids in cases:
        want = []
        for i, g in enumerate(ids):
            if want and g == ids[want[-1][0]] + want[-1][1]:
                want[-1] = (want[-1][0], want[-1][1] + 1)
            else:
                want.append((i, 1))
        assert nk.nk_page_runs(ids) == want
