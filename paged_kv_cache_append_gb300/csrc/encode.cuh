// encode.cuh -- fused quantization of one token-head row (K or V side) into
// its code and scale bytes, shared by the append kernel and the fused
// append + decode kernel.
//
// "Paged KV cache" maintainer design page: the page names the profiles and
// their plane sizes but leaves the codec rules open; the rules implemented
// here are this library's (nk.h, nk_profile):
//   INT8-G64  s = min(fp16(fp32(amax/127)), 65504), q = clamp(RNE(x/s), -127, 127)
//   FP8-row   s = min(fp16(fp32(amax/448)), 65504), c = E4M3FN RNE satfinite (x/s)
//   NVFP4-G16 s8 = E4M3FN RNE satfinite (fp32(amax/6)), c = E2M1 RNE satfinite (x/s8)
// fp32 quotients (__fdiv_rn) followed by one RNE conversion give the exactly
// rounded quotient for these operand widths, so codes are bit-exact.  The
// binary16 scales saturate: RNE rounding is monotone, so clamping the fp32
// quotient at 65504 before the conversion equals clamping the rounded value.
//
// One warp encodes one row: lane i owns elements [i*EL, (i+1)*EL) with
// EL = D/32, so a quantization group of 64 (or 16) elements is a run of
// consecutive lanes and its amax is a shuffle reduction over those lanes.
#pragma once

#include "device.cuh"
#include "internal.h"

namespace nk {

template <int N>
struct Bytes;
template <> struct Bytes<1> { using T = uint8_t; };
template <> struct Bytes<2> { using T = uint16_t; };
template <> struct Bytes<4> { using T = uint32_t; };
template <> struct Bytes<8> { using T = uint2; };
template <> struct Bytes<16> { using T = uint4; };

// Loads EL consecutive bf16 values as floats.
template <int EL>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* p, float* x, typename Bytes<2 * EL>::T& raw) {
  raw = *reinterpret_cast<const typename Bytes<2 * EL>::T*>(p);
  const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
  for (int i = 0; i < EL; ++i) x[i] = __bfloat162float(h[i]);
}

template <int LANES>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int off = 1; off < LANES; off <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Encodes one side (K or V) of one token-head row.  `code_row` / `scale_row`
// point at byte 0 of the row in the code / scale plane.
template <int KIND, int D>
__device__ __forceinline__ void encode_row(const __nv_bfloat16* src, uint8_t* code_row,
                                           uint8_t* scale_row, int lane) {
  constexpr int EL = D / 32;
  float x[EL];
  typename Bytes<2 * EL>::T raw;
  load_bf16<EL>(src + lane * EL, x, raw);
  if constexpr (KIND == KIND_BF16) {
    *reinterpret_cast<typename Bytes<2 * EL>::T*>(code_row + lane * EL * 2) = raw;
  } else if constexpr (KIND == KIND_INT8) {
    constexpr int LPG = 64 / EL;  // lanes per 64-element group
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < EL; ++i) a = fmaxf(a, fabsf(x[i]));
    a = group_max<LPG>(a);
    const __half s = __float2half_rn(fminf(__fdiv_rn(a, 127.f), 65504.f));
    const float sf = __half2float(s);
    uint8_t q[EL];
#pragma unroll
    for (int i = 0; i < EL; ++i) {
      int v = 0;
      if (sf != 0.f) v = max(-127, min(127, __float2int_rn(__fdiv_rn(x[i], sf))));
      q[i] = static_cast<uint8_t>(static_cast<int8_t>(v));
    }
    *reinterpret_cast<typename Bytes<EL>::T*>(code_row + lane * EL) =
        *reinterpret_cast<const typename Bytes<EL>::T*>(q);
    if (lane % LPG == 0)
      *reinterpret_cast<__half*>(scale_row + (lane / LPG) * 2) = s;
  } else if constexpr (KIND == KIND_FP8) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < EL; ++i) a = fmaxf(a, fabsf(x[i]));
    a = group_max<32>(a);
    const __half s = __float2half_rn(fminf(__fdiv_rn(a, 448.f), 65504.f));
    const float sf = __half2float(s);
    uint8_t c[EL];
#pragma unroll
    for (int i = 0; i < EL; i += 2) {
      uint16_t p = 0;
      if (sf != 0.f) p = f32x2_to_e4m3x2(__fdiv_rn(x[i], sf), __fdiv_rn(x[i + 1], sf));
      c[i] = static_cast<uint8_t>(p & 0xFF);
      c[i + 1] = static_cast<uint8_t>(p >> 8);
    }
    *reinterpret_cast<typename Bytes<EL>::T*>(code_row + lane * EL) =
        *reinterpret_cast<const typename Bytes<EL>::T*>(c);
    if (lane == 0) *reinterpret_cast<__half*>(scale_row) = s;
  } else {  // NVFP4-G16
    constexpr int LPG = 16 / EL;  // lanes per 16-element group
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < EL; ++i) a = fmaxf(a, fabsf(x[i]));
    a = group_max<LPG>(a);
    const uint32_t s8 = f32x2_to_e4m3x2(__fdiv_rn(a, 6.f), 0.f) & 0xFFu;
    const float sv = e4m3_to_f32(s8);
    uint8_t c[EL / 2];
#pragma unroll
    for (int i = 0; i < EL; i += 2) {
      uint32_t b = 0;
      if (sv != 0.f) b = f32x2_to_e2m1x2(__fdiv_rn(x[i], sv), __fdiv_rn(x[i + 1], sv));
      c[i / 2] = static_cast<uint8_t>(b);
    }
    *reinterpret_cast<typename Bytes<EL / 2>::T*>(code_row + lane * (EL / 2)) =
        *reinterpret_cast<const typename Bytes<EL / 2>::T*>(c);
    if (lane % LPG == 0) scale_row[lane / LPG] = static_cast<uint8_t>(s8);
  }
}

// Code and scale bytes per token-head row of a profile side.
template <int KIND>
__host__ __device__ constexpr int code_row_bytes(int D) {
  return KIND == KIND_BF16 ? 2 * D : KIND == KIND_NVFP4 ? D / 2 : D;
}
template <int KIND>
__host__ __device__ constexpr int scale_row_bytes(int D) {
  return KIND == KIND_BF16 ? 0 : KIND == KIND_INT8 ? 2 * (D / 64) : KIND == KIND_FP8 ? 2 : D / 16;
}

}  // namespace nk
