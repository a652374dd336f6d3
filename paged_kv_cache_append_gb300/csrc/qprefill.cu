// qprefill.cu -- chunked prefill / replay attention over quantized pages on
// the 5th-generation tensor cores: INT8-G64, FP8-E4M3FN-row256, NVFP4-G16 and
// K8V4 (FP8-row K, NVFP4 V) pools.
//
// The pages are read in place through the block table and dequantized inside
// the attention kernel, page tile by page tile, in shared memory ("Paged KV
// cache" maintainer design page, consumer view: no gather to a contiguous
// cache and no staging copy whose size grows with the context).  One CTA owns
// 128 query rows of one (row b, KV head h), as in the BF16 prefill
// (prefill.cu):
//   warp 4      TMA producer: the raw code tile of each page (the pool's own
//               tensor maps, 64 rows x min(row bytes, 128) boxes) and its
//               scale tile (bulk copy) into a raw K ring and a raw V ring;
//   warps 6-13  converters: each page's codes become an f16 tile in the
//               layout the MMAs read (rows = keys, 128-byte rows of 64 dims,
//               128-byte swizzle), K one page ahead of V; with K they
//               store each key's fp32 factors (K: score factor times
//               softmax_scale * log2 e; V: softmax weight factor) in a
//               small ring of their own;
//   warp 5      MMA issuer: S = Q K^T (A = Q in TMEM, B = the f16 K tile),
//               O += P V (A = P in TMEM, B = the f16 V tile, MN-major);
//   warps 0-3   Q to TMEM (f16, each query row prescaled by a power of two),
//               online softmax with the per-key factors, epilogue.
// Per page the raw codes cross HBM / L2 once per CTA; the f16 tiles never
// leave the SM.
//
// Every operand is exact ("Paged KV cache" page: dequantization belongs to
// the attention consumer; the codec rules are this library's, nk.h):
//   * E4M3 and E2M1 codes are exact binary16 values, and an E2M1 code times
//     its E4M3 group scale is an exact binary16 product (at most 6
//     significant bits, within range), so NVFP4 pages become exact f16 values;
//   * FP8-row pages keep their codes, and the row scale of each key is applied
//     in fp32 to its score (K) and its softmax weight (V);
//   * q is scaled per query row by a power of two, 2^e with max|q| 2^e in
//     [2^14, 2^15), which makes bf16 -> f16 exact for every element above
//     max|q| 2^-31; the scores divide 2^e back out in fp32.
// Every profile rescales lazily (a row's maximum moves only when a score
// passes it by more than 2^8, so p <= 2^8).  FP8-row V weights p * s_key are
// lifted by a power of two 2^K, s_max 2^K in [2^6, 2^7) for the largest V
// scale seen so far (v_lift), so that they stay finite and far from f16's
// subnormal range for V of any magnitude; 2^K is carried by l and O alike and
// leaves with the row's maximum (m - K) in the epilogue.
// INT8-G64 is the one profile whose dequantized values are not f16 values: an
// INT8 code (7 bits) times its binary16 group scale (11 bits) needs up to 18
// significant bits.  A per-key power of two 2^-e, e in [0, 7], keeps the
// largest element of the key below 2^15 (every binary16 scale is at most
// 65504, so every key fits f16); 2^e goes into the key's fp32 factor (K) or
// its softmax weight (V), which stays below 2^8 * 2^7 under the lazy 2^8
// threshold.  With s' = s_g 2^-e as a binary16 value (exact whenever e = 0,
// i.e. every key below 2^15, and otherwise unless the shift takes it below
// binary16's normal range, where the element's error stays under 2^-32 of the
// key's largest element):
//   * keys are exact: each K tile is held as two f16 tiles k1 = f16(c s') and
//     k2' = k1 - c s' (an f16 value, see convert_tile), and S accumulates
//     Q k1^T - Q k2'^T (the second MMA negates its B operand), so the scores
//     are those of the dequantized keys up to the fp32 accumulation;
//   * values are rounded once, c s' to f16 (relative error <= 2^-11 per
//     element, as the f16 softmax weights themselves).
#include <cmath>

#include "encode.cuh"
#include "internal.h"
#include "prefill_split.cuh"
#include "tcgen05.cuh"

namespace nk {

struct QArgs {
  const __nv_bfloat16* q;  // [B][Tc][Hq][D]
  const int32_t* tables;
  const int32_t* table_rows;
  const int32_t* prefix_len;
  const int32_t* chunk_len;
  const uint8_t* ks;  // layer scale planes: K scales, V scales
  const uint8_t* vs;
  __nv_bfloat16* out;
  float* lse;
  int* status;
  float scale_log2;  // softmax_scale * log2(e)
  int B, Tc, Hq, H, G, L, M, C;
  PrefillSplit sp;
  int head_major;  // plane order
};

// INT8-G64 keys: the power of two e (0..7) with 127 * max_g s_g * 2^-e < 2^15
// (or the largest, 7, when binary16's range forbids it).  The scales are
// finite and >= 0, so 127 * max_g s_g is 0 or a normal fp32 x, and
// x < 2^ex for ex = (biased exponent of x) - 126.
template <int D>
__device__ __forceinline__ int int8_row_shift(const uint8_t* scale_row) {
  float smax = 0.f;
#pragma unroll
  for (int g = 0; g < D / 64; ++g)
    smax = fmaxf(smax, fabsf(__half2float(*reinterpret_cast<const __half*>(scale_row + 2 * g))));
  const int ex = static_cast<int>((__float_as_uint(127.f * smax) >> 23) & 0xFFu) - 126;
  return min(max(ex - 15, 0), 7);
}

// 2^-e for e in [0, 7] (a normal fp32).
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

// Rescale threshold of the online softmax, in log2 units: the running maximum
// moves only when a score passes it by more than this, so p <= 2^8.
constexpr float kLazyThr = 8.f;

template <int KK, int KV, int D>
struct QCfg {
  // converter warps (6 .. 5 + NCONV), 8 for every profile: the conversion
  // work sets the pace where only V is converted (raw FP8 keys go to the
  // tensor cores) as well as where both are
  static constexpr int NCONV = 8;
  static constexpr int THREADS = 192 + 32 * NCONV;  // warps 0-3 softmax, 4 producer, 5 MMA
  static constexpr int KCB = code_row_bytes<KK>(D), VCB = code_row_bytes<KV>(D);
  static constexpr int KSB = scale_row_bytes<KK>(D), VSB = scale_row_bytes<KV>(D);
  static constexpr int K_RB = KCB < 128 ? KCB : 128, V_RB = VCB < 128 ? VCB : 128;
  static constexpr int F16 = 64 * D * 2;                           // one f16 page tile
  // INT8-G64 keys are held as two f16 tiles whose sum is exact (K_SPLIT)
  static constexpr bool K_SPLIT = KK == KIND_INT8;
  static constexpr int K_STAGE = K_SPLIT ? 2 * F16 : F16;
  static constexpr int V_STAGE = F16;
  static constexpr int NF = 4;                                     // factor ring (512 B per page)
  static constexpr int RK_CODES = (64 * KCB + 1023) / 1024 * 1024;  // raw K code tile (1024-aligned)
  static constexpr int RV_CODES = (64 * VCB + 1023) / 1024 * 1024;
  static constexpr int RK_STAGE = (RK_CODES + 64 * KSB + 1023) / 1024 * 1024;
  static constexpr int RV_STAGE = (RV_CODES + 64 * VSB + 1023) / 1024 * 1024;
  // FP8-row keys with 128-byte code rows (head_dim >= 128, the swizzle of the
  // f16 tiles) go to the tensor cores as raw E4M3 codes (kind::f8f6f4), with
  // q split exactly into two E4M3 terms: no K conversion, no f16 K tile.
  static constexpr bool K8MMA = (KK == KIND_FP8) && D >= 128;
  static constexpr int NK = K8MMA ? 0 : K_SPLIT ? (D == 256 ? 1 : D == 128 ? 3 : 6)
                                              : D == 256 ? 2 : D == 128 ? 4 : 6;  // f16 K ring
  static constexpr int NV = K8MMA ? (D == 256 ? 3 : 4) : K_SPLIT ? (D == 256 ? 2 : D == 128 ? 3 : 6) : NK;  // f16 V ring
  static constexpr int NRK = K8MMA ? (D == 256 ? 3 : 6) : D == 256 ? (RK_STAGE <= 10240 ? 3 : 2) : 4;  // raw rings
  static constexpr int NRV = D == 256 ? (RV_STAGE <= 10240 || K8MMA ? 3 : 2) : 4;
  static constexpr int NKF = K8MMA ? 0 : NK;  // f16 K ready barriers (the raw FP8 keys need none)
  static constexpr int OFF_V = NK * K_STAGE;
  static constexpr int OFF_RK = OFF_V + NV * V_STAGE;
  static constexpr int OFF_RV = OFF_RK + NRK * RK_STAGE;
  static constexpr int OFF_F = OFF_RV + NRV * RV_STAGE;
  static constexpr int OFF_BAR = OFF_F + NF * 512;
  static constexpr int NBAR = 2 * NKF + 2 * NV + 2 * NRK + 2 * NRV + 2 * NF + 2 + 4;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 64 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0, COL_Q = 128, COL_O = 256;
  static constexpr uint32_t ID_S = K8MMA ? tc::idesc_e4m3(128, 64) : tc::idesc_f16(128, 64, false, false);
  static constexpr uint32_t ID_O = tc::idesc_f16(128, D, false, true);
  static constexpr int UNITS = 64 * (D / 16);  // (key, 16-dim group) units of a tile
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ void q_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Byte address (offset in the raw tile) of byte `col` of key row r in a tile
// staged as blocks of 64 rows x RB bytes with the matching TMA swizzle.
template <int RB>
__device__ __forceinline__ uint32_t raw_off(int r, int col) {
  return static_cast<uint32_t>((col / RB) * (64 * RB)) + swz<RB>(r, col % RB);
}

// Offset of f16 element (key r, dim d) in an f16 tile: 64-dim blocks of
// 64 rows x 128 bytes, 128-byte swizzle (d a multiple of 8: a 16-byte chunk).
__device__ __forceinline__ uint32_t f16_off(int r, int d) {
  return static_cast<uint32_t>((d >> 6) * 8192) + swz<128>(r, (d & 63) * 2);
}

// 16 dims [16 g, 16 g + 16) of key r of an FP8-row or NVFP4-G16 tile: raw
// codes and scales (shared memory) -> 16 exact f16 values (two 16-byte
// chunks).  INT8-G64 tiles are converted in convert_tile.
template <int KIND, int D, int RB>
__device__ __forceinline__ void convert16(const uint8_t* codes, const uint8_t* scales, int r, int g, uint4& lo,
                                          uint4& hi) {
  static_assert(KIND == KIND_FP8 || KIND == KIND_NVFP4, "FP8-row and NVFP4-G16 tiles");
  constexpr int SB = scale_row_bytes<KIND>(D);
  if constexpr (KIND == KIND_FP8) {
    const uint4 w = *reinterpret_cast<const uint4*>(codes + raw_off<RB>(r, 16 * g));
    lo = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w.x & 0xFFFFu)),
                    e4m3x2_to_f16x2(static_cast<uint16_t>(w.x >> 16)),
                    e4m3x2_to_f16x2(static_cast<uint16_t>(w.y & 0xFFFFu)),
                    e4m3x2_to_f16x2(static_cast<uint16_t>(w.y >> 16)));
    hi = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w.z & 0xFFFFu)),
                    e4m3x2_to_f16x2(static_cast<uint16_t>(w.z >> 16)),
                    e4m3x2_to_f16x2(static_cast<uint16_t>(w.w & 0xFFFFu)),
                    e4m3x2_to_f16x2(static_cast<uint16_t>(w.w >> 16)));
  } else {  // NVFP4: 8 bytes of codes times the group's E4M3 scale
    const uint2 w = *reinterpret_cast<const uint2*>(codes + raw_off<RB>(r, 8 * g));
    const uint32_t s16 = e4m3x2_to_f16x2(static_cast<uint16_t>(scales[r * SB + g])) & 0xFFFFu;
    const uint32_t s2 = s16 | (s16 << 16);
    lo = make_uint4(hmul2_u32(e2m1x2_byte_to_f16x2<0>(w.x), s2), hmul2_u32(e2m1x2_byte_to_f16x2<1>(w.x), s2),
                    hmul2_u32(e2m1x2_byte_to_f16x2<2>(w.x), s2), hmul2_u32(e2m1x2_byte_to_f16x2<3>(w.x), s2));
    hi = make_uint4(hmul2_u32(e2m1x2_byte_to_f16x2<0>(w.y), s2), hmul2_u32(e2m1x2_byte_to_f16x2<1>(w.y), s2),
                    hmul2_u32(e2m1x2_byte_to_f16x2<2>(w.y), s2), hmul2_u32(e2m1x2_byte_to_f16x2<3>(w.y), s2));
  }
}

// Factor of key r of a raw tile: FP8-row its row scale, INT8-G64 its 2^e,
// NVFP4 1 (the scales are inside the f16 values).
template <int KIND, int D>
__device__ __forceinline__ float key_factor(const uint8_t* scales, int r) {
  constexpr int SB = scale_row_bytes<KIND>(D);
  if constexpr (KIND == KIND_FP8) return __half2float(*reinterpret_cast<const __half*>(scales + r * SB));
  else if constexpr (KIND == KIND_INT8) return __uint_as_float(static_cast<uint32_t>(127 + int8_row_shift<D>(scales + r * SB)) << 23);
  else return 1.f;
}

// One converter thread's share of a page tile, in units of (key r, 16-dim
// group g): key r = (ct & 7) + 8 ((ct >> 3) & 7) and the UPT groups
// UPT (ct >> 6) + [0, UPT), so every unit of a thread shares its key (the
// INT8 key shift is computed once).  Eight consecutive threads take eight
// consecutive keys of one group, so the swizzled 16-byte loads and stores are
// free of bank conflicts; the next eight threads take their groups one step
// ahead, which keeps the 8-byte NVFP4 loads (16 threads per access) apart.
// NCT, the number of converter threads, is a multiple of 64; keys at or past
// `kvalid` become zeros.
//
// SPLIT (INT8-G64 only): the tile is written twice, as k1 = f16(c s') and, at
// f16 + 64 D 2, as the negated remainder k2' = k1 - c s', with s' = s_g 2^-e
// the binary16 scale.  c s' is a multiple of 2^-24 with at most 7 + 11
// significant bits, so the remainder (at most 7 bits, the same multiple) is an
// f16 value and k1 - k2' = c s' exactly: one f16 FMA per pair, fma(c, -s', k1),
// gives it, and the MMA that reads k2' negates its B operand.
template <int KIND, int D, int RB, int NCT, bool SPLIT = false>
__device__ __forceinline__ void convert_tile(const uint8_t* raw, int raw_codes, uint8_t* f16, int ct, int kvalid) {
  constexpr int GPR = D / 16;            // 16-dim groups per key
  constexpr int UPT = (64 * GPR) / NCT;  // units per thread
  static_assert(UPT * NCT == 64 * GPR && UPT >= 1, "converter units");
  static_assert(!SPLIT || KIND == KIND_INT8, "split tiles are for INT8-G64 keys");
  // a thread's UPT groups start at a multiple of UPT, so with 16 UPT dividing
  // 64 they share one INT8-G64 scale group
  static_assert(KIND != KIND_INT8 || 64 % (16 * UPT) == 0, "one scale group per thread");
  constexpr int SB = scale_row_bytes<KIND>(D);
  const uint8_t* scales = raw + raw_codes;
  const int r = (ct & 7) + 8 * ((ct >> 3) & 7);  // the thread's key
  int gg[UPT];
#pragma unroll
  for (int k = 0; k < UPT; ++k) gg[k] = UPT * (ct >> 6) + (k + ((ct >> 3) & 1)) % UPT;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  if (r >= kvalid) {  // a key at or past the frontier: zeros in every tile
#pragma unroll
    for (int k = 0; k < UPT; ++k) {
      const uint32_t o0 = f16_off(r, 16 * gg[k]), o1 = f16_off(r, 16 * gg[k] + 8);
      *reinterpret_cast<uint4*>(f16 + o0) = zero;
      *reinterpret_cast<uint4*>(f16 + o1) = zero;
      if constexpr (SPLIT) {
        *reinterpret_cast<uint4*>(f16 + 128 * D + o0) = zero;
        *reinterpret_cast<uint4*>(f16 + 128 * D + o1) = zero;
      }
    }
    return;
  }
  if constexpr (KIND == KIND_INT8) {
    // code times the key's shifted binary16 scale s' = s_g 2^-e (once per
    // thread; exact unless the shift takes it below binary16's normal range),
    // the product rounded once (k1); SPLIT also stores the remainder k2
    const float shift = pow2_neg(int8_row_shift<D>(scales + r * SB));
    const __half s16 =
        __float2half_rn(__half2float(*reinterpret_cast<const __half*>(scales + r * SB + 2 * ((16 * gg[0]) / 64))) * shift);
    const uint32_t s2 = pack_h2(s16, s16), s2n = s2 ^ 0x80008000u;  // s', -s'
    // every raw load of the thread before any store (the stores could alias)
    uint4 w[UPT];
#pragma unroll
    for (int k = 0; k < UPT; ++k) w[k] = *reinterpret_cast<const uint4*>(raw + raw_off<RB>(r, 16 * gg[k]));
#pragma unroll
    for (int k = 0; k < UPT; ++k) {
      const uint32_t wv[4] = {w[k].x ^ 0x80808080u, w[k].y ^ 0x80808080u, w[k].z ^ 0x80808080u,
                              w[k].w ^ 0x80808080u};
      uint32_t k1[8], k2[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t c0 = s8pair_flipped_to_f16x2<0>(wv[q]);
        const uint32_t c1 = s8pair_flipped_to_f16x2<1>(wv[q]);
        k1[2 * q] = hmul2_u32(c0, s2);
        k1[2 * q + 1] = hmul2_u32(c1, s2);
        if constexpr (SPLIT) {
          k2[2 * q] = hfma2_u32(c0, s2n, k1[2 * q]);
          k2[2 * q + 1] = hfma2_u32(c1, s2n, k1[2 * q + 1]);
        }
      }
      const uint32_t o0 = f16_off(r, 16 * gg[k]), o1 = f16_off(r, 16 * gg[k] + 8);
      *reinterpret_cast<uint4*>(f16 + o0) = make_uint4(k1[0], k1[1], k1[2], k1[3]);
      *reinterpret_cast<uint4*>(f16 + o1) = make_uint4(k1[4], k1[5], k1[6], k1[7]);
      if constexpr (SPLIT) {
        *reinterpret_cast<uint4*>(f16 + 128 * D + o0) = make_uint4(k2[0], k2[1], k2[2], k2[3]);
        *reinterpret_cast<uint4*>(f16 + 128 * D + o1) = make_uint4(k2[4], k2[5], k2[6], k2[7]);
      }
    }
  } else {
    uint4 lo[UPT], hi[UPT];
    // every raw load of the thread before any store (the stores could alias)
#pragma unroll
    for (int k = 0; k < UPT; ++k) convert16<KIND, D, RB>(raw, scales, r, gg[k], lo[k], hi[k]);
#pragma unroll
    for (int k = 0; k < UPT; ++k) {
      *reinterpret_cast<uint4*>(f16 + f16_off(r, 16 * gg[k])) = lo[k];
      *reinterpret_cast<uint4*>(f16 + f16_off(r, 16 * gg[k] + 8)) = hi[k];
    }
  }
}

template <int KK, int KV, int D>
__global__ void __launch_bounds__((QCfg<KK, KV, D>::THREADS), 1)
    qprefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, QArgs a) {
  using Cfg = QCfg<KK, KV, D>;
  constexpr int NK = Cfg::NK, NV = Cfg::NV, NRK = Cfg::NRK, NRV = Cfg::NRV, NF = Cfg::NF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + Cfg::OFF_V;
  uint8_t* sRK = smem + Cfg::OFF_RK;
  uint8_t* sRV = smem + Cfg::OFF_RV;
  float* sF = reinterpret_cast<float*>(smem + Cfg::OFF_F);  // [NF][128]: 64 K factors, 64 V factors
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  constexpr int NKF = Cfg::NKF;
  uint64_t* k_full = bars;             // f16 K tile ready for the MMA (converters)
  uint64_t* k_empty = k_full + NKF;    // S of the f16 tile done (MMA commit; f16 K only)
  uint64_t* v_full = k_empty + NKF;    // f16 V tile ready (converters)
  uint64_t* v_empty = v_full + NV;     // PV of the tile done (MMA commit)
  uint64_t* rk_full = v_empty + NV;    // raw K tile landed (TMA)
  uint64_t* rk_empty = rk_full + NRK;  // raw K tile consumed
  uint64_t* rv_full = rk_empty + NRK;
  uint64_t* rv_empty = rv_full + NRV;
  uint64_t* f_full = rv_empty + NRV;  // factors of a page written (converters)
  uint64_t* f_empty = f_full + NF;    // factors read (softmax warps)
  uint64_t* s_full = f_empty + NF;    // [2]
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* q_ready = o_done + 1;
  uint64_t* drain = q_ready + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* s_last = s_abort + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x / a.sp.nsplit, split = blockIdx.x % a.sp.nsplit;
  const int h = blockIdx.y, b = blockIdx.z;
  const int G = a.G, TQ = 128 / G;
  griddep_wait();  // launched with programmatic stream serialization
  griddep_launch_dependents();

  const int row = a.table_rows[b];
  const int prefix = a.prefix_len[b], chunk = a.chunk_len[b];
  if (row < 0 || row >= a.C || prefix < 0 || chunk < 0 || chunk > a.Tc ||
      static_cast<int64_t>(prefix) + chunk > static_cast<int64_t>(a.L) * 64) {
    if (tid == 0 && qt == 0 && h == 0) set_status(a.status, NK_STATUS_FRONTIER);
    return;
  }
  const int t0 = qt * TQ;
  if (t0 >= chunk) return;
  const int t_last = min(t0 + TQ, chunk) - 1;
  const int nkt = (prefix + t_last + 1 + 63) / 64;
  // this split's pages [p_lo, p_lo + n); local page i is absolute page p_lo + i
  const int per = (nkt + a.sp.nsplit - 1) / a.sp.nsplit;
  const int p_lo = min(split * per, nkt);
  const int n = min(p_lo + per, nkt) - p_lo;
  const int F = prefix + chunk;  // keys >= F of a page are stale
  const int32_t* table = a.tables + static_cast<int64_t>(row) * a.L + p_lo;

  if (tid == 0) {
    for (int i = 0; i < NKF; ++i) {
      mbar_init(&k_full[i], Cfg::NCONV);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&v_full[i], Cfg::NCONV);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < NRK; ++i) {
      mbar_init(&rk_full[i], 1);
      // released by the converters; with raw FP8 keys also by the MMA commit
      mbar_init(&rk_empty[i], Cfg::K8MMA ? 1 + Cfg::NCONV : Cfg::NCONV);
    }
    for (int i = 0; i < NRV; ++i) {
      mbar_init(&rv_full[i], 1);
      mbar_init(&rv_empty[i], Cfg::NCONV);
    }
    for (int i = 0; i < NF; ++i) {
      mbar_init(&f_full[i], Cfg::NCONV);
      mbar_init(&f_empty[i], 4);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(q_ready, 4);
    mbar_init(drain, 1);
    *s_abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  if (warp == 0) {
    tc::alloc(tslot, Cfg::TMEM_COLS);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 4) {
    // ------------- TMA producer: raw code and scale tiles of each page -----------
    int gnext = 0;
    for (int j = 0; j < n; ++j) {
      if ((j & 31) == 0) gnext = (j + lane < n) ? table[j + lane] : 0;
      int g = __shfl_sync(0xffffffffu, gnext, j & 31);
      int stop = 0;
      if (lane == 0) {
        if (g < 0 || g >= a.M) {  // never copy from outside the pool
          set_status(a.status, NK_STATUS_PAGE_RANGE);
          g = 0;
        }
        const int y = static_cast<int>(tile_row(g, h, a.H, a.M, a.head_major));
        const int rk = j % NRK, rv = j % NRV;
        if (j >= NRK && !mbar_wait_bounded(&rk_empty[rk], ((j / NRK) - 1) & 1, a.status)) stop = 1;
        if (!stop) {
          uint8_t* st = sRK + rk * Cfg::RK_STAGE;
          mbar_arrive_expect_tx(&rk_full[rk], 64 * Cfg::KCB + 64 * Cfg::KSB);
#pragma unroll
          for (int c = 0; c < Cfg::KCB / Cfg::K_RB; ++c)
            tma_load_2d(st + c * 64 * Cfg::K_RB, &tmk, c * Cfg::K_RB, y, &rk_full[rk]);
          bulk_load(st + Cfg::RK_CODES, a.ks + static_cast<int64_t>(y) * Cfg::KSB, 64 * Cfg::KSB, &rk_full[rk]);
        }
        if (!stop && j >= NRV && !mbar_wait_bounded(&rv_empty[rv], ((j / NRV) - 1) & 1, a.status)) stop = 1;
        if (!stop) {
          uint8_t* st = sRV + rv * Cfg::RV_STAGE;
          mbar_arrive_expect_tx(&rv_full[rv], 64 * Cfg::VCB + 64 * Cfg::VSB);
#pragma unroll
          for (int c = 0; c < Cfg::VCB / Cfg::V_RB; ++c)
            tma_load_2d(st + c * 64 * Cfg::V_RB, &tmv, c * Cfg::V_RB, y, &rv_full[rv]);
          bulk_load(st + Cfg::RV_CODES, a.vs + static_cast<int64_t>(y) * Cfg::VSB, 64 * Cfg::VSB, &rv_full[rv]);
        }
        if (stop) *s_abort = 1;
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) break;
    }
  } else if (warp >= 6) {
    // ------------- converters: K one page ahead of V ------------------------------
    // Order K(0), K(1), V(0), K(2), V(1), ...: the MMA issues S(i) before
    // PV(i - 1).  With K(i) the converters also write page i's per-key
    // factors (K from the K scales, V from the V scales, whose raw tile was
    // loaded with the K tile) into the factor ring, so the softmax of a page
    // never waits for its V tile.
    const int ct = tid - 192;  // 0 .. 32 NCONV - 1
    bool ok = true;
    for (int i = 0; ok && i <= n; ++i) {
      if (i < n) {  // K(i) and the factors of page i
        const int rk = i % NRK, rv = i % NRV, fs = i % NF;
        ok = mbar_wait_bounded(&rk_full[rk], (i / NRK) & 1, a.status) && !*s_abort;
        if (!ok) break;
        const uint8_t* raw = sRK + rk * Cfg::RK_STAGE;
        const int kvalid = F - 64 * (p_lo + i);
        const bool live = ct < 64 && ct < kvalid;
        // key ct's K factor, read before the raw slot can be released
        const float kf = live ? key_factor<KK, D>(raw + Cfg::RK_CODES, ct) * a.scale_log2 : 0.f;
        if constexpr (!Cfg::K8MMA) {
          const int ks = i % NK;
          if (i >= NK) ok = mbar_wait_bounded(&k_empty[ks], ((i / NK) - 1) & 1, a.status) && !*s_abort;
          if (!ok) break;
          convert_tile<KK, D, Cfg::K_RB, 32 * Cfg::NCONV, Cfg::K_SPLIT>(raw, Cfg::RK_CODES, sK + ks * Cfg::K_STAGE, ct,
                                                                       kvalid);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            q_arrive(&rk_empty[rk]);
            q_arrive(&k_full[ks]);
          }
        }
        ok = mbar_wait_bounded(&rv_full[rv], (i / NRV) & 1, a.status) && !*s_abort;
        if (ok && i >= NF) ok = mbar_wait_bounded(&f_empty[fs], ((i / NF) - 1) & 1, a.status) && !*s_abort;
        if (!ok) break;
        if (ct < 64) {
          float* fac = sF + fs * 128;
          fac[ct] = kf;
          fac[64 + ct] = live ? key_factor<KV, D>(sRV + rv * Cfg::RV_STAGE + Cfg::RV_CODES, ct) : 0.f;
        }
        __syncwarp();
        if (lane == 0) {
          q_arrive(&f_full[fs]);
          // the raw E4M3 tile is the MMA operand itself: the slot is free once
          // these scale reads and S(i) (the MMA's commit) are both done
          if constexpr (Cfg::K8MMA) q_arrive(&rk_empty[rk]);
        }
      }
      if (i >= 1) {  // V(i - 1)
        const int jj = i - 1, rv = jj % NRV, vs = jj % NV;
        ok = mbar_wait_bounded(&rv_full[rv], (jj / NRV) & 1, a.status) && !*s_abort;
        if (ok && jj >= NV) ok = mbar_wait_bounded(&v_empty[vs], ((jj / NV) - 1) & 1, a.status) && !*s_abort;
        if (!ok) break;
        convert_tile<KV, D, Cfg::V_RB, 32 * Cfg::NCONV>(sRV + rv * Cfg::RV_STAGE, Cfg::RV_CODES, sV + vs * Cfg::V_STAGE, ct,
                                       F - 64 * (p_lo + jj));
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          q_arrive(&rv_empty[rv]);
          q_arrive(&v_full[vs]);
        }
      }
    }
    if (!ok) *s_abort = 1;
  } else if (warp == 5) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      bool ok = mbar_wait_bounded(q_ready, 0, a.status);
      tc::fence_after();
      for (int j = 0; ok && j <= n; ++j) {
        if (j < n) {  // S(j) = Q K(j)^T into buffer j & 1
          const int sb = j & 1;
          if constexpr (Cfg::K8MMA) {
            // E4M3 codes (32 per instruction: 32 bytes of a 128-byte row, as
            // 16 f16 values are), q_hi in columns [COL_Q, COL_Q + D/4), q_lo
            // in the next D/4
            const int rk = j % NRK;
            ok = mbar_wait_bounded(&rk_full[rk], (j / NRK) & 1, a.status) && !*s_abort;
            if (!ok) break;
            tc::fence_after();
            const uint64_t kd = tc::smem_desc(smem_u32(sRK + rk * Cfg::RK_STAGE), 16, 1024);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
              for (int kk = 0; kk < D / 32; ++kk)
                tc::mma_ts_f8(tmem + Cfg::COL_S + 64 * sb, tmem + Cfg::COL_Q + part * (D / 4) + kk * 8,
                              kd + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), Cfg::ID_S,
                              part > 0 || kk > 0);
            tc::commit(&s_full[sb]);
            tc::commit(&rk_empty[rk]);
          } else {
            const int ks = j % NK;
            ok = mbar_wait_bounded(&k_full[ks], (j / NK) & 1, a.status) && !*s_abort;
            if (!ok) break;
            tc::fence_after();
            // INT8-G64: S = Q k1^T - Q k2'^T from the two f16 tiles of the
            // split keys (the second MMA negates its B operand)
#pragma unroll
            for (int part = 0; part < (Cfg::K_SPLIT ? 2 : 1); ++part) {
              const uint64_t kd = tc::smem_desc(smem_u32(sK + ks * Cfg::K_STAGE + part * Cfg::F16), 16, 1024);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                tc::mma_ts(tmem + Cfg::COL_S + 64 * sb, tmem + Cfg::COL_Q + kk * 8,
                           kd + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4),
                           part > 0 ? tc::idesc_negate_b(Cfg::ID_S) : Cfg::ID_S, part > 0 || kk > 0);
            }
            tc::commit(&s_full[sb]);
            tc::commit(&k_empty[ks]);
          }
        }
        if (j >= 1) {  // O += P(j - 1) V(j - 1)
          const int jj = j - 1, vs = jj % NV;
          ok = mbar_wait_bounded(&v_full[vs], (jj / NV) & 1, a.status) && !*s_abort;
          if (ok) ok = mbar_wait_bounded(p_full, jj & 1, a.status) && !*s_abort;
          if (!ok) break;
          tc::fence_after();
          const uint64_t vd = tc::smem_desc(smem_u32(sV + vs * Cfg::V_STAGE), 8192, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_ts(tmem + Cfg::COL_O, tmem + Cfg::COL_S + 64 * (jj & 1) + kk * 8,
                       vd + static_cast<uint64_t>((kk * 2048) >> 4), Cfg::ID_O, (jj > 0 || kk > 0));
          tc::commit(o_done);
          tc::commit(&v_empty[vs]);
        }
      }
      if (!ok) *s_abort = 1;
      tc::commit(drain);
    }
  } else {
    // ------------------------------ softmax warps -----------------------------
    const int m = tid;
    const int tl = m / G, g = m % G;
    const int token = t0 + tl;
    const bool row_valid = token < chunk;
    const int pos = prefix + token;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float rs = 1.f;  // 2^-e of this query row
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + ((static_cast<int64_t>(b) * a.Tc + token) * a.Hq + h * G + g) * D);
      float mx = 0.f;
      if (row_valid)
        for (int u = 0; u < D / 8; ++u) {
          const uint4 x = src[u];
          const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&x);
#pragma unroll
          for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fabsf(__bfloat162float(e[k])));
        }
      int ex = 0;
      if (mx > 0.f) frexpf(mx, &ex);
      // f16 q: max|q| 2^e in [2^14, 2^15); E4M3 q: max|q| 2^e in [2^7, 2^8)
      const int e = mx > 0.f ? min((Cfg::K8MMA ? 8 : 15) - ex, 100) : 0;  // 2^e stays finite in fp32
      const float qf = ldexpf(1.f, e);
      rs = ldexpf(1.f, -e);
      if constexpr (Cfg::K8MMA) {
        // q' = q 2^e = hi + lo with hi = E4M3(q') and lo = E4M3(q' - hi), both
        // round to nearest even.  Where |q'| >= 2^-2 the residual is an exact
        // E4M3 value (q' has 8 significant bits, hi keeps 4, the rest fit
        // 4 more within E4M3's range), so hi + lo = q'; smaller elements are
        // kept to 2^-10 absolute, i.e. 2^-17 max|q'|.  A 32-bit column holds
        // 4 consecutive dims, the lowest in its low byte.
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t hv[16], lv[16];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = row_valid ? src[c0 / 8 + u] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            uint32_t hpair[4], lpair[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
              const float x0 = __low2float(v) * qf, x1 = __high2float(v) * qf;
              const uint16_t h2 = f32x2_to_e4m3x2(x0, x1);
              const uint32_t hb32 = e4m3x2_to_f16x2(h2);
              const __half2 hb = *reinterpret_cast<const __half2*>(&hb32);
              hpair[k] = h2;
              lpair[k] = f32x2_to_e4m3x2(x0 - __low2float(hb), x1 - __high2float(hb));
            }
            hv[2 * u] = hpair[0] | (hpair[1] << 16);
            hv[2 * u + 1] = hpair[2] | (hpair[3] << 16);
            lv[2 * u] = lpair[0] | (lpair[1] << 16);
            lv[2 * u + 1] = lpair[2] | (lpair[3] << 16);
          }
          tc::st16(tmem + lane_base + Cfg::COL_Q + c0 / 4, hv);
          tc::st16(tmem + lane_base + Cfg::COL_Q + D / 4 + c0 / 4, lv);
        }
      } else {
#pragma unroll 1
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          uint32_t qv[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = row_valid ? src[c0 / 4 + u] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
              qv[4 * u + k] = pack_f16x2(__low2float(v) * qf, __high2float(v) * qf);
            }
          }
          tc::st32(tmem + lane_base + Cfg::COL_Q + c0, qv);
        }
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) q_arrive(q_ready);
    }
    float m_used = -INFINITY, l = 0.f;
    int k_run = KV == KIND_FP8 ? kVLiftInit : 0;  // FP8-row V: the weights, l and O carry 2^k_run (v_lift)
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int sb = j & 1, fs = j % NF;
      ok = mbar_wait_bounded(&s_full[sb], (j / 2) & 1, a.status) && !*s_abort;
      if (ok) ok = mbar_wait_bounded(&f_full[fs], (j / NF) & 1, a.status) && !*s_abort;
      if (!ok) break;
      tc::fence_after();
      uint32_t v0[32], v1[32];
      tc::ld32(tmem + lane_base + Cfg::COL_S + 64 * sb, v0);
      tc::ld32(tmem + lane_base + Cfg::COL_S + 64 * sb + 32, v1);
      tc::wait_ld();
      const float* ksc = sF + fs * 128;
      const float* vsc = ksc + 64;
      const int kmax = row_valid ? pos - 64 * (p_lo + j) : -1;
      // Score factors: per key for FP8-row (row scale) and INT8-G64 (2^e)
      // keys; NVFP4 keys carry their scales in the f16 values, so every key
      // has the plain softmax scale.  The causal mask is applied only where
      // the page reaches past a row's last key.
      constexpr bool KEY_FAC = KK != KIND_NVFP4;
      const bool nomask = __all_sync(0xffffffffu, kmax >= 63);
      float rmax = -INFINITY;
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        float ka[4] = {a.scale_log2, a.scale_log2, a.scale_log2, a.scale_log2}, kb[4] = {ka[0], ka[1], ka[2], ka[3]};
        if constexpr (KEY_FAC) {
          const float4 k0 = *reinterpret_cast<const float4*>(ksc + 4 * c4);
          const float4 k1 = *reinterpret_cast<const float4*>(ksc + 32 + 4 * c4);
          ka[0] = k0.x, ka[1] = k0.y, ka[2] = k0.z, ka[3] = k0.w;
          kb[0] = k1.x, kb[1] = k1.y, kb[2] = k1.z, kb[3] = k1.w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = 4 * c4 + u;
          float x = __uint_as_float(v0[c]) * ka[u], y = __uint_as_float(v1[c]) * kb[u];
          if (!nomask) {
            x = c <= kmax ? x : -INFINITY;
            y = 32 + c <= kmax ? y : -INFINITY;
          }
          v0[c] = __float_as_uint(x);
          v1[c] = __float_as_uint(y);
          rmax = fmaxf(rmax, fmaxf(x, y));
        }
      }
      rmax = rmax == -INFINITY ? -INFINITY : rmax * rs;
      // Weight factors: FP8-row V (row scale) and INT8-G64 V (2^e); NVFP4 V
      // carries its scales in the f16 values.
      constexpr bool VAL_FAC = KV != KIND_NVFP4;
      // FP8-row V: the lift of the largest row scale so far (every lane
      // reads two of the page's 64 scales; the maximum crosses the warp)
      int knew = k_run;
      if constexpr (KV == KIND_FP8) {
        const float2 s2 = *reinterpret_cast<const float2*>(vsc + 2 * lane);
        knew = v_lift(__reduce_max_sync(0xffffffffu, __float_as_uint(fmaxf(s2.x, s2.y))), k_run);
      }
      // p = 2^(z - m + K): a rescale when the maximum passes the lazy
      // threshold or the lift drops
      float factor = 1.f;
      const float mnew = fmaxf(m_used, rmax);
      bool resc = false;
      if (mnew != -INFINITY && (m_used == -INFINITY || mnew > m_used + kLazyThr || knew != k_run)) {
        factor = m_used == -INFINITY ? 0.f : ex2((m_used - mnew) + static_cast<float>(knew - k_run));
        m_used = mnew;
        resc = true;
      }
      k_run = knew;
      const float mu = m_used == -INFINITY ? 0.f : m_used - static_cast<float>(k_run);
      uint32_t pk[32];
      float sum = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        float sa[4] = {1.f, 1.f, 1.f, 1.f}, sbv[4] = {1.f, 1.f, 1.f, 1.f};
        if constexpr (VAL_FAC) {
          const float4 s0 = *reinterpret_cast<const float4*>(vsc + 4 * c4);
          const float4 s1 = *reinterpret_cast<const float4*>(vsc + 32 + 4 * c4);
          sa[0] = s0.x, sa[1] = s0.y, sa[2] = s0.z, sa[3] = s0.w;
          sbv[0] = s1.x, sbv[1] = s1.y, sbv[2] = s1.z, sbv[3] = s1.w;
        }
        float p0[4], p1[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          p0[u] = ex2(fmaf(__uint_as_float(v0[4 * c4 + u]), rs, -mu));
          p1[u] = ex2(fmaf(__uint_as_float(v1[4 * c4 + u]), rs, -mu));
          sum += p0[u] + p1[u];
        }
        if constexpr (VAL_FAC) {
          pk[2 * c4] = pack_f16x2(p0[0] * sa[0], p0[1] * sa[1]);
          pk[2 * c4 + 1] = pack_f16x2(p0[2] * sa[2], p0[3] * sa[3]);
          pk[16 + 2 * c4] = pack_f16x2(p1[0] * sbv[0], p1[1] * sbv[1]);
          pk[16 + 2 * c4 + 1] = pack_f16x2(p1[2] * sbv[2], p1[3] * sbv[3]);
        } else {
          pk[2 * c4] = pack_f16x2(p0[0], p0[1]);
          pk[2 * c4 + 1] = pack_f16x2(p0[2], p0[3]);
          pk[16 + 2 * c4] = pack_f16x2(p1[0], p1[1]);
          pk[16 + 2 * c4 + 1] = pack_f16x2(p1[2], p1[3]);
        }
      }
      __syncwarp();
      if (lane == 0) q_arrive(&f_empty[fs]);  // this warp is done with the page's factors
      l = l * factor + sum;
      if (j >= 1) {
        ok = mbar_wait_bounded(o_done, (j - 1) & 1, a.status) && !*s_abort;
        if (!ok) break;
        tc::fence_after();
      }
      if (__any_sync(0xffffffffu, resc && j >= 1)) {
        const float f = (resc && j >= 1) ? factor : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          tc::ld32(tmem + lane_base + Cfg::COL_O + c0, ov);
          tc::wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * f);
          tc::st32(tmem + lane_base + Cfg::COL_O + c0, ov);
        }
      }
      tc::st32(tmem + lane_base + Cfg::COL_S + 64 * sb, pk);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) q_arrive(p_full);
    }
    if (ok && n > 0) ok = mbar_wait_bounded(o_done, (n - 1) & 1, a.status) && !*s_abort;
    tc::fence_after();
    if (ok) {
      const int64_t orow = (static_cast<int64_t>(b) * a.Tc + token) * a.Hq + h * G + g;
      const int64_t tile = (static_cast<int64_t>(b) * a.H + h) * a.sp.tiles + qt;
      const float m_eff = m_used == -INFINITY ? -INFINITY : m_used - static_cast<float>(k_run);
      prefill_store<D>(tmem + lane_base + Cfg::COL_O, n > 0, row_valid, m_eff, l, a.out + orow * D,
                       a.lse ? a.lse + orow : nullptr, a.sp, tile, split, m, s_last);
    }
  }

  // ---- teardown: every issued MMA has completed before TMEM is freed ---------
  if (warp < 4 && tid == 0) mbar_wait_bounded(drain, 0, a.status, 200000000ull);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::dealloc(tmem, Cfg::TMEM_COLS);
}

template <int KK, int KV, int D>
static cudaError_t launch_q(const CUtensorMap& tk, const CUtensorMap& tv, const QArgs& a, cudaStream_t s) {
  using Cfg = QCfg<KK, KV, D>;
  auto k = qprefill_kernel<KK, KV, D>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(k, dim3(a.sp.tiles * a.sp.nsplit, a.H, a.B), dim3(Cfg::THREADS), Cfg::SMEM, s, tk, tv, a);
}

template <int KK, int KV>
static cudaError_t launch_qd(int D, const CUtensorMap& tk, const CUtensorMap& tv, const QArgs& a, cudaStream_t s) {
  return D == 256   ? launch_q<KK, KV, 256>(tk, tv, a, s)
         : D == 128 ? launch_q<KK, KV, 128>(tk, tv, a, s)
                    : launch_q<KK, KV, 64>(tk, tv, a, s);
}

// Quantized-pool prefill.  The caller (nk_paged_prefill_attention) has checked
// shapes, pointers and alignment; the workspace holds only the split partials.
int qprefill_launch(const nk_pool* p, int layer, const void* q, const int32_t* tables, const int32_t* table_rows,
                    const int32_t* prefix_len, const int32_t* chunk_len, int B, int Tc, int Hq, float scale_log2,
                    void* out, float* lse, void* ws, size_t ws_bytes, cudaStream_t s) {
  const int D = p->desc.head_dim, H = p->desc.num_kv_heads;
  const int tiles = (Tc + 128 / (Hq / H) - 1) / (128 / (Hq / H));
  const int nsplit = prefill_nsplit(tiles * H * B, p->num_sms);
  const size_t need = prefill_split_bytes(B, H, tiles, nsplit, D);
  if (need && (!ws || ws_bytes < need))
    return fail(NK_ERR_WORKSPACE, "workspace needs " + std::to_string(need) + " bytes");
  if (need && !aligned16(ws)) return fail(NK_ERR_ALIGN, "workspace must be 16-byte aligned");
  QArgs a;
  const int np = p->n_planes;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.tables = tables;
  a.table_rows = table_rows;
  a.prefix_len = prefix_len;
  a.chunk_len = chunk_len;
  a.ks = static_cast<const uint8_t*>(p->ptrs[layer * np + 2]);
  a.vs = static_cast<const uint8_t*>(p->ptrs[layer * np + 3]);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.status = p->status;
  a.scale_log2 = scale_log2;
  a.B = B;
  a.Tc = Tc;
  a.Hq = Hq;
  a.H = H;
  a.G = Hq / H;
  a.L = p->L;
  a.M = p->M;
  a.C = p->desc.max_concurrency;
  a.sp = prefill_split_at(ws, B, H, tiles, nsplit);
  a.head_major = p->desc.order == NK_HEAD_MAJOR;
  const CUtensorMap& tk = p->tmap[layer * 2 + 0];
  const CUtensorMap& tv = p->tmap[layer * 2 + 1];
  cudaError_t e;
  switch (p->desc.profile) {
    case NK_INT8_G64: e = launch_qd<KIND_INT8, KIND_INT8>(D, tk, tv, a, s); break;
    case NK_FP8_E4M3_ROW: e = launch_qd<KIND_FP8, KIND_FP8>(D, tk, tv, a, s); break;
    case NK_NVFP4_G16: e = launch_qd<KIND_NVFP4, KIND_NVFP4>(D, tk, tv, a, s); break;
    case NK_K8V4: e = launch_qd<KIND_FP8, KIND_NVFP4>(D, tk, tv, a, s); break;
    default: return fail(NK_ERR_UNSUPPORTED, "no quantized prefill for this profile");
  }
  if (e != cudaSuccess) return cuda_fail(e, "quantized prefill launch");
  return NK_OK;
}

}  // namespace nk
