"""Pins of oracle.codec: exact-rational brute force, invariants, page byte table."""

import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import codec, formats as F, layout
from tests.exact_rounding import (e2m1_nearest_code, e4m3_nearest_code, round_rational,
                                  to_fp16, to_fp32)
from tests.test_oracle_formats import _e4m3_exact_table

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_vectors(rng, n, D, outliers=True, lo=-3, hi=3):
    x = rng.standard_normal((n, D))
    if outliers:
        x *= np.where(rng.random((n, D)) < 0.02, 20.0, 1.0)
    x *= 10.0 ** rng.integers(lo, hi, (n, 1))
    return F.f64_to_bf16_bits(x)


def test_byte_table_matches_page():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "byte_table_d256.txt"))
            if l.strip() and not l.startswith("#")]
    assert [r[0] for r in rows] == list(layout.PROFILES)
    for name, kc, ks, vc, vs, tot in rows:
        sch = {p.name: p.row_bytes for p in layout.plane_schema(name, 256)}
        assert sch.get("k") == int(kc) and sch.get("v") == int(vc)
        assert sch.get("k_scale", 0) == int(ks) and sch.get("v_scale", 0) == int(vs)
        assert layout.bytes_per_token_head(name, 256) == int(tot)
    # the asymmetric K8V4 total is not 2 * vector_bytes of either side
    assert layout.bytes_per_token_head("k8v4", 256) not in (2 * 258, 2 * 144)


# ------------------------------------------------- exact-rational brute force

def test_int8_g64_brute_force():
    rng = np.random.default_rng(10)
    bits = _bf16_vectors(rng, 40, 128)
    x = F.bf16_bits_to_f64(bits)
    q, sb = codec.int8_g64_quant(x)
    s = F.fp16_from_bits(sb)
    for r in range(x.shape[0]):
        for g in range(2):
            xs = [Fraction(float(v)) for v in x[r, 64 * g:64 * g + 64]]
            amax = max(abs(v) for v in xs)
            s_ref = to_fp16(to_fp32(amax / 127))
            assert Fraction(float(s[r, g])) == s_ref
            for j, v in enumerate(xs):
                want = 0 if s_ref == 0 else max(-127, min(127, round(v / s_ref)))
                assert int(q[r, 64 * g + j]) == want


def test_fp8_row_brute_force():
    rng = np.random.default_rng(11)
    table = _e4m3_exact_table()
    bits = _bf16_vectors(rng, 12, 64)
    x = F.bf16_bits_to_f64(bits)
    c, sb = codec.fp8_row_quant(x)
    for r in range(x.shape[0]):
        xs = [Fraction(float(v)) for v in x[r]]
        s_ref = to_fp16(to_fp32(max(abs(v) for v in xs) / 448))
        assert Fraction(float(F.fp16_from_bits(sb[r, 0]))) == s_ref
        for j, v in enumerate(xs):
            want = e4m3_nearest_code(v / s_ref, bool(np.signbit(x[r, j])), table)
            assert int(c[r, j]) == want


def test_nvfp4_g16_brute_force():
    rng = np.random.default_rng(12)
    table = _e4m3_exact_table()
    bits = _bf16_vectors(rng, 12, 64)
    x = F.bf16_bits_to_f64(bits)
    packed, s8 = codec.nvfp4_g16_quant(x)
    c = codec.nvfp4_unpack(packed)
    for r in range(x.shape[0]):
        for g in range(4):
            xs = [Fraction(float(v)) for v in x[r, 16 * g:16 * g + 16]]
            amax = max(abs(v) for v in xs)
            s_code = e4m3_nearest_code(to_fp32(amax / 6), False, table)
            assert int(s8[r, g]) == s_code
            sv = dict(table)[s_code]
            for j, v in enumerate(xs):
                if sv == 0:
                    want = 0
                else:
                    want = e2m1_nearest_code(v / sv, bool(np.signbit(x[r, 16 * g + j])))
                assert int(c[r, 16 * g + j]) == want


def test_float64_quotient_is_exact_rounding():
    """The claim the codec docstring makes: RNE of a float64 quotient x/s
    equals RNE of the exact quotient for bf16 x and binary16 s."""
    rng = np.random.default_rng(13)
    xb = F.bf16_bits_to_f64(rng.integers(0, 0x7F80, 3000, dtype=np.uint16))
    sb = F.fp16_from_bits(rng.integers(1, 0x7C00, 3000, dtype=np.uint16))
    for x, s in zip(xb, sb):
        q64 = x / s
        exact = Fraction(float(x)) / Fraction(float(s))
        assert int(np.clip(np.rint(q64), -127, 127)) == max(-127, min(127, round(exact)))
        assert Fraction(float(F.e4m3_round(q64))) == min(round_rational(exact, 3, -6), 448)


# ------------------------------------------------------------- invariants

@pytest.mark.parametrize("kind", ["int8_g64", "fp8_row", "nvfp4_g16"])
def test_amax_element_maps_to_format_max(kind):
    rng = np.random.default_rng(14)
    x = F.bf16_bits_to_f64(_bf16_vectors(rng, 200, 256, lo=-1, hi=2))
    grp = {"int8_g64": 64, "fp8_row": 256, "nvfp4_g16": 16}[kind]
    xg = x.reshape(200, -1, grp)
    idx = np.argmax(np.abs(xg), axis=-1)
    if kind == "int8_g64":
        q, _ = codec.int8_g64_quant(x)
        top = np.take_along_axis(q.reshape(200, -1, grp).astype(int), idx[..., None], -1)[..., 0]
        sign = np.sign(np.take_along_axis(xg, idx[..., None], -1)[..., 0])
        assert np.all(top == 127 * sign)
    elif kind == "fp8_row":
        c, _ = codec.fp8_row_quant(x)
        top = np.take_along_axis(c.reshape(200, -1, grp), idx[..., None], -1)[..., 0]
        assert np.all((top & 0x7F) == 0x7E)
    else:
        p, s8 = codec.nvfp4_g16_quant(x)
        c = codec.nvfp4_unpack(p).reshape(200, -1, grp)
        top = np.take_along_axis(c, idx[..., None], -1)[..., 0]
        live = (s8 >= 0x08) & (s8 != 0x7E)      # normal, unsaturated E4M3 scale
        assert np.all((top[live] & 7) == 7)


@pytest.mark.parametrize("kind", ["int8_g64", "fp8_row", "nvfp4_g16"])
def test_requantize_is_idempotent(kind):
    """quant(dequant(codes)) returns the same codes and scales (no scale
    saturation or subnormal scale in this data)."""
    rng = np.random.default_rng(15)
    x = F.bf16_bits_to_f64(_bf16_vectors(rng, 64, 256, lo=-1, hi=1))
    quant = {"int8_g64": codec.int8_g64_quant, "fp8_row": codec.fp8_row_quant,
             "nvfp4_g16": codec.nvfp4_g16_quant}[kind]
    dequant = {"int8_g64": codec.int8_g64_dequant, "fp8_row": codec.fp8_row_dequant,
               "nvfp4_g16": codec.nvfp4_g16_dequant}[kind]
    c, s = quant(x)
    c2, s2 = quant(dequant(c, s))
    assert np.array_equal(c, c2) and np.array_equal(s, s2)


def test_int8_error_bound():
    rng = np.random.default_rng(16)
    x = F.bf16_bits_to_f64(_bf16_vectors(rng, 100, 256, outliers=False))
    q, sb = codec.int8_g64_quant(x)
    xh = codec.int8_g64_dequant(q, sb)
    s = np.repeat(F.fp16_from_bits(sb), 64, axis=-1)
    unclamped = np.abs(q.astype(int)) < 127
    assert np.all(np.abs(x - xh)[unclamped] <= s[unclamped] / 2)


def test_fp8_error_bound():
    rng = np.random.default_rng(17)
    x = F.bf16_bits_to_f64(_bf16_vectors(rng, 100, 256, outliers=False))
    c, sb = codec.fp8_row_quant(x)
    xh = codec.fp8_row_dequant(c, sb)
    s = F.fp16_from_bits(sb)
    u = x / s
    # half an E4M3 ulp at |u| (quantum 2**(max(e,-6)-3)), times s
    e = np.maximum(np.floor(np.log2(np.maximum(np.abs(u), 2.0 ** -20))), -6)
    assert np.all(np.abs(u - xh / s) <= 2.0 ** (e - 3) / 2 + 1e-12)


def test_zero_and_tiny_groups():
    x = np.zeros((1, 64))
    q, sb = codec.int8_g64_quant(x)
    assert not q.any() and not sb.any()
    c, sb = codec.fp8_row_quant(x)
    assert not c.any() and not sb.any()
    tiny = np.full((1, 16), 1e-3)            # amax/6 rounds to E4M3 zero
    p, s8 = codec.nvfp4_g16_quant(tiny)
    assert not s8.any() and not p.any()
    neg0 = np.array([[1.0] + [-0.0] * 63])
    c, _ = codec.fp8_row_quant(neg0)
    assert c[0, 0] == 0x7E and np.all(c[0, 1:] == 0x80)


def test_binary16_scales_saturate():
    """Closed forms above the binary16 range: amax / 127 (or / 448) past the
    largest finite binary16 leaves s = 65504, the amax element takes the
    extreme code, an exact multiple of s keeps its exact code, and every
    dequantized value is finite.  Just below the edge the scale is the plain
    rounded quotient."""
    for amax in (253 * 32768.0, 254 * 32768.0, 2.0 ** 26, 3.0e38):
        x = np.zeros((1, 64))
        x[0, 5], x[0, 9] = -amax, 3 * 65504.0
        q, sb = codec.int8_g64_quant(x)
        s = F.fp16_from_bits(sb)[0, 0]
        if amax / 127 < 65504:
            assert s == 65280.0                       # 253 * 32768 / 127 = 65278 -> 65280
            assert q[0, 5] == -127
        else:
            assert s == 65504.0
            assert q[0, 5] == -127 and q[0, 9] == 3
        assert np.all(np.isfinite(codec.int8_g64_dequant(q, sb)))
    for amax in (2.0 ** 26, 3.0e38):
        x = np.zeros((1, 128))
        x[0, 0], x[0, 1] = amax, -2 * 65504.0
        c, sb = codec.fp8_row_quant(x)
        assert F.fp16_from_bits(sb)[0, 0] == 65504.0
        assert c[0, 0] == 0x7E and c[0, 1] == 0xC0    # +448 (saturated), -2.0
        assert np.all(np.isfinite(codec.fp8_row_dequant(c, sb)))


def test_nibble_order_low_first():
    x = np.zeros((1, 16))
    x[0, 0], x[0, 1] = 6.0, -3.0             # scale 1.0 -> codes 7 and 0xD
    p, s8 = codec.nvfp4_g16_quant(x)
    assert F.e4m3_decode(s8)[0, 0] == 1.0
    assert p[0, 0] == 0x7 | (0xD << 4)
