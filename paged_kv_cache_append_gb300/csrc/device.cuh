// device.cuh -- sm_103a device helpers shared by the libnk kernels:
// mbarrier with bounded waits, TMA / bulk-async copies, ldmatrix, warp-level
// mma.sync, and the narrow-format conversions of the KV codecs.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "nk.h"

namespace nk {

// Kernels OR NK_STATUS_* bits into the device status word whose address the
// host passes them (see status_word() in pool.cu); nk_status_read() reads it.
__device__ __forceinline__ void set_status(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// --------------------------------------------- programmatic dependent launch

// Waits until the grids this one depends on have completed and flushed their
// memory (no-op when the launch had no programmatic dependency).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next grid in the stream start launching (its own griddep_wait still
// waits for this grid to complete).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` with programmatic stream serialization, so its CTAs may
// start while the previous kernel in the stream drains.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; gives up after
// `limit_ns` of wall time, records NK_STATUS_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status,
                                                  uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      set_status(status, NK_STATUS_TIMEOUT);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------ async copies

// L2 prefetch of `bytes` (a multiple of 16) at a 16-byte aligned address.  L2
// is the point of coherence, so a prefetch issued before a dependency wait
// cannot make a later load return stale data.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// 2-D tiled TMA load: box at (x = column, y = row) of the tensor map.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------ ldmatrix / mma

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), fp32 accumulate.
template <bool BF16>
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// ------------------------------------------------------------ conversions

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^k as a float, for -126 <= k <= 127 (exact).
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float(static_cast<uint32_t>(127 + k) << 23); }

// ------------------------------------------------------------ FP8-row V lift
// Kernels that apply FP8-row value scales to the softmax weights store
// p * s_key as f16 operands of P V, with p <= 2^8 (the lazy rescale
// threshold).  Raw, p * s would leave f16's normal range for small V (s is
// amax / 448) and overflow for V near the binary16 limit.  The weights are
// therefore lifted by a power of two 2^K chosen from the largest scale s_max
// seen so far, s_max 2^K in [2^6, 2^7): every lifted weight stays below 2^15
// and the large ones far above the subnormal range, whatever the magnitude
// of V.  K only decreases along a row's keys (the accumulators are rescaled
// when it does) and starts at kVLiftInit, the value for the smallest positive
// binary16 scale, 2^-24.
constexpr int kVLiftTop = 6, kVLiftInit = kVLiftTop + 24, kVLiftMin = kVLiftTop - 15;

// K after a tile whose largest value scale has the bits smax_bits (a
// non-negative float; 0 when every scale of the tile is zero: K stays).  K is
// at least kVLiftMin, the value for the largest binary16 scale, 65504.
__device__ __forceinline__ int v_lift(uint32_t smax_bits, int k_run) {
  if (smax_bits == 0u) return k_run;
  return min(k_run, max(kVLiftTop + 127 - static_cast<int>(smax_bits >> 23), kVLiftMin));
}

// Two E4M3FN codes (low byte = element 0) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Byte I of w (two E2M1 codes, low nibble = element 0) -> f16x2 (exact).
#define NK_E2M1_BYTE(SEL)                                  \
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"                     \
      " mov.b32 {b0, b1, b2, b3}, %1;\n"                   \
      " cvt.rn.f16x2.e2m1x2 %0, " SEL ";\n}"               \
      : "=r"(r)                                            \
      : "r"(w))
template <int I>
__device__ __forceinline__ uint32_t e2m1x2_byte_to_f16x2(uint32_t w) {
  uint32_t r;
  if constexpr (I == 0) NK_E2M1_BYTE("b0");
  else if constexpr (I == 1) NK_E2M1_BYTE("b1");
  else if constexpr (I == 2) NK_E2M1_BYTE("b2");
  else NK_E2M1_BYTE("b3");
  return r;
}
#undef NK_E2M1_BYTE

// f32 pair -> two E4M3FN codes, RNE, satfinite; `lo` goes to the low byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// f32 pair -> one byte of two E2M1 codes, RNE, satfinite; `lo` in the low nibble.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n .reg .b8 b;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n"
      " mov.b32 %0, {b, 0, 0, 0};\n}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// One E4M3FN code -> float (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  return __half2float(__ushort_as_half(static_cast<uint16_t>(e4m3x2_to_f16x2(code & 0xFFu))));
}

// Four signed int8 codes in w: bytes (b0, b1) -> f16x2 exact values.
// (1024 + (b ^ 0x80)) is built in the binary16 mantissa, then 1152 is
// subtracted: 1024 + 128 + b - 1152 = b, exact in binary16.
__device__ __forceinline__ uint32_t s8pair_to_f16x2(uint32_t w_pair_in_bytes_0_2) {
  const uint32_t x =
      (w_pair_in_bytes_0_2 & 0x00FF00FFu) ^ 0x64806480u;  // bytes 1,3 <- 0x64, bytes 0,2 ^ 0x80
  const __half2 h = *reinterpret_cast<const __half2*>(&x);
  const __half2 r = __hsub2(h, __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// The same from a word whose sign bits were flipped already (w ^ 0x80808080,
// once per four codes): the pair (b_2k, b_2k+1) of the word -> f16x2, built
// by one byte permute against the 0x64 exponent bytes.
template <int K>
__device__ __forceinline__ uint32_t s8pair_flipped_to_f16x2(uint32_t w_flipped) {
  static_assert(K == 0 || K == 1, "pair 0 (bytes 0, 1) or 1 (bytes 2, 3)");
  const uint32_t x = __byte_perm(w_flipped, 0x64646464u, K == 0 ? 0x4140 : 0x4342);
  const __half2 h = *reinterpret_cast<const __half2*>(&x);
  const __half2 r = __hsub2(h, __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// a * b + c on f16x2, rounded once
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b),
                      *reinterpret_cast<const __half2*>(&c));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
  __half2 h = __halves2half2(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte address inside a TMA-swizzled tile whose rows are `RB` bytes
// (RB in {32, 64, 128}): 16-byte chunk index bits [4, 4+log2(RB/16)) are
// XORed with address bits [7, 7+...), i.e. the CU_TENSOR_MAP_SWIZZLE_{32,64,128}B
// pattern on a 1024-byte aligned tile.
template <int RB>
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t col) {
  const uint32_t off = row * RB + col;
  return off ^ (((off >> 7) & (RB / 16 - 1)) << 4);
}

}  // namespace nk
