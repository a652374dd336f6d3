"""Exact scalar number formats (test infrastructure only).

The KV profiles named by the "Paged KV cache" design page (page-major plane
layout section: BF16, INT8-G64, FP8-E4M3FN-row256, NVFP4-G16, K8V4) store
codes in small binary formats.  This module rounds an exactly known real
number (held in float64) to those formats with IEEE round-to-nearest,
ties-to-even, and maps values to their bit codes.

Formats (sign, exponent bits, fraction bits, smallest normal exponent):

* binary16 (fp16):      1, 5, 10, e_min = -14; overflow rounds to +-inf.
* E4M3FN (OCP FP8):     1, 4, 3,  e_min = -6; largest finite 448; the code
                        S.1111.111 is NaN; no infinities.  ``satfinite``
                        clamps to +-448.
* E2M1 (OCP FP4):       1, 2, 1,  e_min = 0; values {0, .5, 1, 1.5, 2, 3, 4, 6};
                        ``satfinite`` clamps to +-6.

``round_binary`` works on the exact value: a float64 holding a value |v| in
[2**e, 2**(e+1)) is divided by the power of two 2**(max(e, e_min) - frac_bits)
(exact), rounded to an integer with ``numpy.rint`` (ties to even) and scaled
back (exact).  Pinned by tests: against numpy's float32->float16 cast (a
library routine) and against an exhaustive nearest-neighbour search over every
finite code of E4M3FN / E2M1.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_to_f64", "f64_to_bf16_bits", "round_binary", "round_fp16",
    "fp16_bits", "fp16_from_bits", "E4M3_VALUES", "E2M1_VALUES",
    "e4m3_round", "e4m3_encode", "e4m3_decode", "e2m1_round", "e2m1_encode",
    "e2m1_decode", "fp32",
]

E4M3_MAX = 448.0
E2M1_MAX = 6.0
FP16_MAX = 65504.0


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bfloat16 (ties to even) and return the bits.

    Used only to build inputs and to round oracle outputs the way a bf16
    store would; the rounding goes through ``round_binary`` with 7 fraction
    bits and the float32 exponent range.
    """
    r = round_binary(np.asarray(x, dtype=np.float64), frac_bits=7, e_min=-126)
    r32 = r.astype(np.float32)          # exact: r has 8 significant bits
    return (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def fp32(x) -> np.ndarray:
    """Round to IEEE binary32 (numpy's float64 -> float32 cast, RNE)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def round_binary(v, frac_bits: int, e_min: int) -> np.ndarray:
    """Round exact values ``v`` to a binary format with ``frac_bits`` fraction
    bits and smallest normal exponent ``e_min``; unbounded above (the caller
    applies overflow or saturation).  Ties go to the even significand.  The
    sign of ``v`` is kept, so a negative value that rounds to zero gives -0.0.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                 # a = m * 2**ex, m in [0.5, 1)
    e = np.maximum(ex - 1, e_min)       # a in [2**e, 2**(e+1)) for normals
    quantum = np.ldexp(1.0, (e - frac_bits).astype(np.int32))
    r = np.rint(a / quantum) * quantum  # a / quantum is exact (power of two)
    return np.copysign(r, v)


# ---------------------------------------------------------------- binary16

def round_fp16(v) -> np.ndarray:
    """IEEE binary16 round-to-nearest-even; overflow gives +-inf."""
    r = round_binary(v, frac_bits=10, e_min=-14)
    return np.where(np.abs(r) > FP16_MAX, np.copysign(np.inf, r), r)


def fp16_bits(v_exact_fp16) -> np.ndarray:
    """Bits of values that are already exactly representable in binary16."""
    return np.asarray(v_exact_fp16, dtype=np.float64).astype(np.float16).view(np.uint16)


def fp16_from_bits(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


# ------------------------------------------------------------- E4M3FN

def _e4m3_table() -> np.ndarray:
    vals = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = s * (m / 8.0) * 2.0 ** -6
        else:
            vals[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


E4M3_VALUES = _e4m3_table()             # decode table indexed by code
_E4M3_POS = E4M3_VALUES[:0x7F]          # codes 0x00..0x7E, strictly increasing


def e4m3_round(v) -> np.ndarray:
    """E4M3FN round-to-nearest-even with satfinite (clamp to +-448)."""
    r = round_binary(v, frac_bits=3, e_min=-6)
    return np.where(np.abs(r) > E4M3_MAX, np.copysign(E4M3_MAX, r), r)


def e4m3_encode(v) -> np.ndarray:
    """Exact value -> E4M3FN code (RNE, satfinite).  The code's sign bit is the
    sign of ``v`` (so -0.0 and small negatives that round to zero give 0x80)."""
    r = e4m3_round(v)
    mag = np.searchsorted(_E4M3_POS, np.abs(r))
    assert np.all(_E4M3_POS[mag] == np.abs(r))
    sign = np.signbit(r).astype(np.uint8) << np.uint8(7)
    return (mag.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


# ---------------------------------------------------------------- E2M1

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                        -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def e2m1_round(v) -> np.ndarray:
    """E2M1 round-to-nearest-even with satfinite (clamp to +-6)."""
    r = round_binary(v, frac_bits=1, e_min=0)
    return np.where(np.abs(r) > E2M1_MAX, np.copysign(E2M1_MAX, r), r)


def e2m1_encode(v) -> np.ndarray:
    """Exact value -> 4-bit E2M1 code in 0..15 (sign in bit 3)."""
    r = e2m1_round(v)
    mag = np.searchsorted(E2M1_VALUES[:8], np.abs(r))
    assert np.all(E2M1_VALUES[mag] == np.abs(r))
    sign = np.signbit(r).astype(np.uint8) << np.uint8(3)
    return (mag.astype(np.uint8) | sign).astype(np.uint8)


def e2m1_decode(codes) -> np.ndarray:
    return E2M1_VALUES[np.asarray(codes, dtype=np.uint8) & 0xF]
