"""Pins of oracle.formats against things other than itself."""

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F
from tests.exact_rounding import e2m1_nearest_code, e4m3_nearest_code, round_rational


def _fp16_grid_ties():
    """Midpoints between adjacent binary16 values (exact in float32)."""
    h = np.arange(0, 0x7C00, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    nxt = np.nextafter(h.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    return ((h + nxt) / 2)[np.isfinite(nxt)]


def test_round_fp16_matches_numpy_cast():
    rng = np.random.default_rng(0)
    mag = np.ldexp(rng.uniform(1, 2, 20000), rng.integers(-30, 17, 20000))
    x32 = (mag * rng.choice([-1, 1], mag.size)).astype(np.float32)
    extra = np.array([0.0, -0.0, 65504, 65519.99, 65520, 65536, 6.0e-8, 2.0 ** -25,
                      2.0 ** -24, 3 * 2.0 ** -25, 2.0 ** -14, 1e-10], dtype=np.float32)
    ties = _fp16_grid_ties().astype(np.float32)
    x32 = np.concatenate([x32, extra, -extra, ties, -ties])
    want = x32.astype(np.float16).astype(np.float64)        # library routine
    got = F.round_fp16(x32.astype(np.float64))
    assert np.array_equal(np.signbit(got), np.signbit(want))
    assert np.array_equal(got, want)


def test_fp16_rounding_matches_exact_rationals():
    rng = np.random.default_rng(1)
    xs = np.ldexp(rng.uniform(1, 2, 400), rng.integers(-28, 16, 400))
    for x in xs:
        want = round_rational(Fraction(float(x)), 10, -14)
        assert Fraction(float(F.round_fp16(x))) == want


def test_bf16_bits_known_values():
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000, 0x4049], dtype=np.uint16)
    want = [1.0, -2.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, -0.0, 3.140625]
    got = F.bf16_bits_to_f64(bits)
    assert list(got) == want
    assert np.signbit(got[4])


def test_f64_to_bf16_matches_torch_cast():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-5, 5, 5000),
                        [0.0, -0.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8]])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.f64_to_bf16_bits(x), want)


def test_e4m3_table_spec_values():
    # OCP FP8 E4M3FN: bias 7, no infinities, S.1111.111 is NaN.
    assert F.E4M3_VALUES[0x7E] == 448.0
    assert F.E4M3_VALUES[0xFE] == -448.0
    assert F.E4M3_VALUES[0x01] == 2.0 ** -9
    assert F.E4M3_VALUES[0x08] == 2.0 ** -6
    assert F.E4M3_VALUES[0x38] == 1.0
    assert F.E4M3_VALUES[0x3C] == 1.5
    assert np.isnan(F.E4M3_VALUES[0x7F]) and np.isnan(F.E4M3_VALUES[0xFF])
    pos = F.E4M3_VALUES[:0x7F]
    assert np.all(np.diff(pos) > 0)


def _e4m3_exact_table():
    out = []
    for c in range(0x7F):
        e, m = (c >> 3) & 0xF, c & 7
        if e == 0:
            val = Fraction(m, 8) * Fraction(2) ** -6
        else:
            val = (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        out.append((c, val))
    return out


def test_e4m3_encode_exhaustive_nearest():
    table = _e4m3_exact_table()
    vals = [v for _, v in table]
    samples = [Fraction(0)]
    for a, b in zip(vals[:-1], vals[1:]):         # every tie and its neighbours
        mid = (a + b) / 2
        samples += [mid, mid + (b - a) / 64, mid - (b - a) / 64]
    samples += [Fraction(448), Fraction(460), Fraction(464), Fraction(470), Fraction(10 ** 6)]
    rng = np.random.default_rng(3)
    samples += [Fraction(float(x)) for x in np.ldexp(rng.uniform(1, 2, 3000), rng.integers(-14, 10, 3000))]
    for s in samples:
        for neg in (False, True):
            v = -s if neg else s
            got = int(F.e4m3_encode(-float(s) if neg else float(s)))
            assert got == e4m3_nearest_code(v, neg, table), (s, neg)


def test_e2m1_ties_and_saturation():
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
             0.0: 0, 6.0: 7, 7.0: 7, 100.0: 7, 0.24: 0, 0.26: 1}
    for v, code in cases.items():
        assert int(F.e2m1_encode(v)) == code, v
        assert int(F.e2m1_encode(-v)) == code | 8, v
    # value of the tie cases: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    assert list(F.e2m1_decode(F.e2m1_encode([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]))) == \
        [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_e2m1_encode_exhaustive_nearest():
    rng = np.random.default_rng(4)
    xs = np.concatenate([rng.uniform(0, 8, 4000), np.arange(0, 7.0, 0.125)])
    for x in xs:
        for neg in (False, True):
            got = int(F.e2m1_encode(-x if neg else x))
            assert got == e2m1_nearest_code(Fraction(float(x)), neg), (x, neg)


def test_negative_zero_codes():
    assert int(F.e4m3_encode(-0.0)) == 0x80
    assert int(F.e4m3_encode(-1e-9)) == 0x80
    assert int(F.e4m3_encode(0.0)) == 0x00
    assert int(F.e2m1_encode(-0.1)) == 0x8
    assert int(F.e2m1_encode(-0.0)) == 0x8


@pytest.mark.parametrize("frac,emin", [(23, -126), (10, -14), (3, -6), (1, 0)])
def test_round_binary_matches_exact_rationals(frac, emin):
    rng = np.random.default_rng(5 + frac)
    xs = np.ldexp(rng.uniform(1, 2, 500), rng.integers(emin - 6, 12, 500)) * rng.choice([-1, 1], 500)
    for x in xs:
        got = Fraction(float(F.round_binary(x, frac, emin)))
        assert got == round_rational(Fraction(float(x)), frac, emin)
