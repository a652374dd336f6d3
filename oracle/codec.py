"""Persistent KV codecs of the five profiles (test infrastructure only).

The "Paged KV cache" design page names the profiles and fixes their plane
shapes and byte sizes (page-major layout section and the D256 byte table),
but not their scale or rounding rules.  This library states its own rules, and
both the oracle (here) and the CUDA append kernel are held to them.  ``x``
below is one token's vector for one KV head (D bf16 values, exact in
float64); "RNE" is round to nearest, ties to even; a quotient is the exact
quotient rounded once.

BF16        codes are the bf16 bits, stored unchanged (no fp16 conversion on
            write, as the page requires for the BF16 profile).
INT8-G64    per group of 64 elements along d:
              amax = max|x|;  s = min(fp16(fp32(amax / 127)), 65504)  (fp32
              quotient, then binary16 RNE, saturating at the largest finite
              binary16);  q = clamp(RNE(x / s), -127, 127);
              s == 0 gives q = 0.  Scale plane: binary16 bits.
FP8-row     one scale per (token, head) row of D elements:
              s = min(fp16(fp32(amax / 448)), 65504);
              c = E4M3FN_RNE_satfinite(x / s);
              s == 0 gives c = 0x00.  Scale plane: binary16 bits.
NVFP4-G16   per group of 16 elements along d:
              s8 = E4M3FN_RNE_satfinite(fp32(amax / 6))  (an E4M3 byte);
              c = E2M1_RNE_satfinite(x / decode(s8)); s8 == 0 gives c = 0;
              element 2i goes to the low nibble, 2i+1 to the high nibble of
              byte i.  No per-tensor global scale.
K8V4        K uses FP8-row, V uses NVFP4-G16 (closed asymmetric profile).

The binary16 scales saturate (a reading: the page fixes no overflow rule,
and the E4M3 / E2M1 codes saturate too): without it a group with amax above
127 * 65504 (or 448 * 65504) would store s = +inf and dequantize to NaN.

A code's sign bit is the sign of the quotient, so -0.0 and negative values
that round to zero encode as 0x80 (E4M3) or 0x8 (E2M1).  INT8 has no -0.

Why float64 quotients give the exactly rounded result: x has 8 significant
bits and s at most 11; a quotient that is not itself a rounding tie of the
target format lies at least 2**-16 (relative) away from every tie, far more
than the 2**-53 error of a float64 quotient.  The tests check this claim with
exact rational arithmetic (``fractions.Fraction``).

Pinned by: idempotence quant(dequant(c)) == c; the amax element maps to
+-127 / +-448 / +-6; |x - dequant| bounds; exact-rational brute force on
small inputs; the E2M1/E4M3 tie cases.
"""

from __future__ import annotations

import numpy as np

from . import formats as F


def _fp32_div(a, b) -> np.ndarray:
    """IEEE binary32 quotient of two float64 values exact in binary32."""
    return (F.fp32(a) / np.float32(b)).astype(np.float64)


# ---------------------------------------------------------------- INT8-G64

def int8_g64_quant(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """x [..., D] float64 -> (codes int8 [..., D], scale bits uint16 [..., D/64])."""
    D = x.shape[-1]
    g = x.reshape(*x.shape[:-1], D // 64, 64)
    amax = np.max(np.abs(g), axis=-1)
    s = np.minimum(F.round_fp16(_fp32_div(amax, 127.0)), F.FP16_MAX)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(g / s[..., None])
    q = np.where(s[..., None] == 0, 0.0, np.clip(q, -127, 127))
    return q.reshape(x.shape).astype(np.int8), F.fp16_bits(s)


def int8_g64_dequant(codes: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    D = codes.shape[-1]
    s = F.fp16_from_bits(scale_bits)
    g = codes.astype(np.float64).reshape(*codes.shape[:-1], D // 64, 64)
    return (g * s[..., None]).reshape(codes.shape)


# ---------------------------------------------------------------- FP8-row

def fp8_row_quant(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """x [..., D] -> (E4M3 codes uint8 [..., D], scale bits uint16 [..., 1])."""
    amax = np.max(np.abs(x), axis=-1, keepdims=True)
    s = np.minimum(F.round_fp16(_fp32_div(amax, 448.0)), F.FP16_MAX)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = x / s
    c = F.e4m3_encode(np.where(s == 0, 0.0, v))
    return c, F.fp16_bits(s)


def fp8_row_dequant(codes: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    return F.e4m3_decode(codes) * F.fp16_from_bits(scale_bits)


# -------------------------------------------------------------- NVFP4-G16

def nvfp4_g16_quant(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """x [..., D] -> (packed codes uint8 [..., D/2], E4M3 scales uint8 [..., D/16])."""
    D = x.shape[-1]
    g = x.reshape(*x.shape[:-1], D // 16, 16)
    amax = np.max(np.abs(g), axis=-1)
    s8 = F.e4m3_encode(_fp32_div(amax, 6.0))
    sv = F.e4m3_decode(s8)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = g / sv[..., None]
    c = F.e2m1_encode(np.where(sv[..., None] == 0, 0.0, v)).reshape(x.shape)
    packed = (c[..., 0::2] | (c[..., 1::2] << np.uint8(4))).astype(np.uint8)
    return packed, s8


def nvfp4_unpack(packed: np.ndarray) -> np.ndarray:
    lo = packed & np.uint8(0xF)
    hi = packed >> np.uint8(4)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def nvfp4_g16_dequant(packed: np.ndarray, s8: np.ndarray) -> np.ndarray:
    c = F.e2m1_decode(nvfp4_unpack(packed))
    D = c.shape[-1]
    sv = F.e4m3_decode(s8)
    g = c.reshape(*c.shape[:-1], D // 16, 16) * sv[..., None]
    return g.reshape(c.shape)


# ------------------------------------------------------------ per profile

def _as_bytes(a: np.ndarray) -> np.ndarray:
    """Little-endian byte view of the last axis."""
    a = np.ascontiguousarray(a)
    return a.view(np.uint8).reshape(*a.shape[:-1], a.shape[-1] * a.dtype.itemsize)


def _vector_planes(kind: str, x_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray | None]:
    """Encode one side (K or V) with a vector codec -> (code bytes, scale bytes)."""
    if kind == "bf16":
        return _as_bytes(np.asarray(x_bits, dtype=np.uint16)), None
    x = F.bf16_bits_to_f64(x_bits)
    if kind == "int8_g64":
        c, s = int8_g64_quant(x)
        return _as_bytes(c.view(np.uint8)), _as_bytes(s)
    if kind == "fp8_row":
        c, s = fp8_row_quant(x)
        return c, _as_bytes(s)
    if kind == "nvfp4_g16":
        c, s = nvfp4_g16_quant(x)
        return c, s
    raise ValueError(kind)


def _vector_decode(kind: str, code_bytes: np.ndarray, scale_bytes) -> np.ndarray:
    if kind == "bf16":
        bits = np.ascontiguousarray(code_bytes).view(np.uint16)
        return F.bf16_bits_to_f64(bits)
    if kind == "int8_g64":
        s = np.ascontiguousarray(scale_bytes).view(np.uint16)
        return int8_g64_dequant(np.ascontiguousarray(code_bytes).view(np.int8), s)
    if kind == "fp8_row":
        s = np.ascontiguousarray(scale_bytes).view(np.uint16)
        return fp8_row_dequant(code_bytes, s)
    if kind == "nvfp4_g16":
        return nvfp4_g16_dequant(code_bytes, scale_bytes)
    raise ValueError(kind)


def side_kinds(profile: str) -> tuple[str, str]:
    """Vector codec of the K side and of the V side of a profile."""
    if profile == "k8v4":
        return "fp8_row", "nvfp4_g16"
    return profile, profile


def encode_kv(profile: str, k_bits: np.ndarray, v_bits: np.ndarray) -> dict[str, np.ndarray]:
    """Quantize K and V vectors (bf16 bits [..., D]) into per-plane byte rows
    {plane name: uint8 [..., row_bytes]}."""
    kk, vk = side_kinds(profile)
    kc, ks = _vector_planes(kk, k_bits)
    vc, vs = _vector_planes(vk, v_bits)
    out = {"k": kc, "v": vc}
    if ks is not None:
        out["k_scale"] = ks
        out["v_scale"] = vs
    return out


def decode_kv(profile: str, rows: dict[str, np.ndarray]) -> tuple[np.ndarray, np.ndarray]:
    """Per-plane byte rows -> dequantized (K, V) float64 [..., D]."""
    kk, vk = side_kinds(profile)
    k = _vector_decode(kk, rows["k"], rows.get("k_scale"))
    v = _vector_decode(vk, rows["v"], rows.get("v_scale"))
    return k, v
