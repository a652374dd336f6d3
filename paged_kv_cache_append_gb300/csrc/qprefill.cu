// qprefill.cu -- chunked prefill / replay attention over quantized pages on
// the 5th-generation tensor cores: INT8-G64, FP8-E4M3FN-row256, NVFP4-G16 and
// K8V4 (FP8-row K, NVFP4 V) pools.
//
// Two launches, split by what bounds them:
//   1. qdequant_kernel (HBM bound) converts each page of the prefill rows
//      once into an f16 scratch in logical page order, with per-key fp32
//      scales; pages past a row's frontier are not touched, rows past it are
//      zero.  Every CTA of the tensor pass would otherwise re-convert the same
//      pages (128 query rows share each page), which made the conversion,
//      not the tensor cores, the bound.
//   2. qprefill_kernel (tensor bound) is the BF16 prefill (prefill.cu) on
//      f16 operands: K and V page tiles come from the scratch by TMA, Q and P
//      live in TMEM, and the per-key scales multiply the fp32 scores (K) and
//      the softmax weights (V).
// Every operand is exact ("Paged KV cache" page: dequantization belongs to
// the attention consumer; the codec rules are this library's, nk.h):
//   * E4M3 and E2M1 codes are exact binary16 values, and an E2M1 code times
//     its E4M3 group scale is an exact binary16 product (at most 6
//     significant bits, within range), so NVFP4 pages become exact f16 values;
//   * FP8-row pages keep their codes, and the row scale of each key is applied
//     in fp32;
//   * q is scaled per query row by a power of two, 2^e with max|q| 2^e in
//     [2^14, 2^15), which makes bf16 -> f16 exact for every element above
//     max|q| 2^-31; the scores divide 2^e back out in fp32.
// With FP8-row V the weights p * s_key must stay finite in f16, so the running
// maximum is exact (p <= 1); NVFP4 V keeps the lazy 2^8 rescale threshold.
// INT8-G64 is the one profile whose dequantized values are not exact in f16:
// an INT8 code (7 bits) times its binary16 group scale (11 bits) needs up to
// 18 significant bits, and an exact form would need one fp32 accumulator per
// 64-dim group of each key, four times the S columns of tensor memory.  Its
// pages are dequantized as code * s_g computed exactly in fp32 and rounded
// once to f16 (relative error <= 2^-11 per element), after a per-key power
// of two 2^-e, e in [0, 7], that keeps the largest element of the key below
// 2^15; 2^e goes into the key's fp32 factor (K) or its softmax weight (V),
// which stays below 2^8 * 2^7 under the lazy 2^8 threshold.  Scores then
// differ from the exact ones by at most 2^-11 of sum_d |q_d k_d| times the
// softmax scale, well inside the attention tolerances.
//
// Scratch (the call's workspace): K f16 [B][H][L][64][D], V f16 likewise,
// scales fp32 [B][H][L][128] (64 K scales times softmax_scale * log2 e, then
// 64 V scales; 0 for keys past the frontier).
#include <cmath>

#include "encode.cuh"
#include "internal.h"
#include "prefill_split.cuh"
#include "tcgen05.cuh"

namespace nk {

struct QScratch {
  __half* k;
  __half* v;
  float* sc;
  static size_t bytes(int B, int H, int L, int D) {
    const size_t pages = static_cast<size_t>(B) * H * L;
    return pages * 64 * D * 2 * 2 + pages * 128 * 4;
  }
  static QScratch at(void* ws, int B, int H, int L, int D) {
    const size_t pages = static_cast<size_t>(B) * H * L;
    char* p = static_cast<char*>(ws);
    return QScratch{reinterpret_cast<__half*>(p), reinterpret_cast<__half*>(p + pages * 64 * D * 2),
                    reinterpret_cast<float*>(p + pages * 64 * D * 4)};
  }
};

struct QArgs {
  const __nv_bfloat16* q;  // [B][Tc][Hq][D]
  const int32_t* tables;
  const int32_t* table_rows;
  const int32_t* prefix_len;
  const int32_t* chunk_len;
  const uint8_t* kc;  // layer planes: K codes, V codes, K scales, V scales
  const uint8_t* vc;
  const uint8_t* ks;
  const uint8_t* vs;
  QScratch scr;
  __nv_bfloat16* out;
  float* lse;
  int* status;
  float scale_log2;  // softmax_scale * log2(e)
  float thr;         // rescale threshold in log2 units
  int B, Tc, Hq, H, G, L, M, C;
  PrefillSplit sp;
  int head_major;  // plane order
};

// Row geometry shared by both passes; false when the row is malformed.
__device__ __forceinline__ bool q_row(const QArgs& a, int b, int& row, int& prefix, int& chunk) {
  row = a.table_rows[b];
  prefix = a.prefix_len[b];
  chunk = a.chunk_len[b];
  return !(row < 0 || row >= a.C || prefix < 0 || chunk < 0 || chunk > a.Tc ||
           static_cast<int64_t>(prefix) + chunk > static_cast<int64_t>(a.L) * 64);
}

// INT8-G64 rows: the power of two e (0..7) with 127 * max_g s_g * 2^-e < 2^15.
template <int D>
__device__ __forceinline__ int int8_row_shift(const uint8_t* scale_row) {
  float smax = 0.f;
#pragma unroll
  for (int g = 0; g < D / 64; ++g)
    smax = fmaxf(smax, fabsf(__half2float(*reinterpret_cast<const __half*>(scale_row + 2 * g))));
  int ex = 0;
  frexpf(127.f * smax, &ex);  // 127 * smax < 2^ex
  return min(max(ex - 15, 0), 7);
}

// 8 dims [d, d + 8) of one token-head row -> 8 f16 values (16 bytes): exact
// for FP8 and NVFP4; for INT8-G64, code * s_g * 2^-e rounded once.
template <int KIND, int D>
__device__ __forceinline__ uint4 dequant8(const uint8_t* code_row, const uint8_t* scale_row, int d) {
  if constexpr (KIND == KIND_INT8) {
    const uint2 w = *reinterpret_cast<const uint2*>(code_row + d);
    const float sg = ldexpf(__half2float(*reinterpret_cast<const __half*>(scale_row + 2 * (d / 64))),
                            -int8_row_shift<D>(scale_row));
    const int8_t* c = reinterpret_cast<const int8_t*>(&w);
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = pack_f16x2(static_cast<float>(c[2 * i]) * sg, static_cast<float>(c[2 * i + 1]) * sg);
    return make_uint4(h[0], h[1], h[2], h[3]);
  } else if constexpr (KIND == KIND_FP8) {
    const uint2 w = *reinterpret_cast<const uint2*>(code_row + d);
    return make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w.x & 0xFFFFu)),
                      e4m3x2_to_f16x2(static_cast<uint16_t>(w.x >> 16)),
                      e4m3x2_to_f16x2(static_cast<uint16_t>(w.y & 0xFFFFu)),
                      e4m3x2_to_f16x2(static_cast<uint16_t>(w.y >> 16)));
  } else {  // NVFP4: 4 bytes of codes times the group's E4M3 scale
    const uint32_t w = *reinterpret_cast<const uint32_t*>(code_row + d / 2);
    const uint32_t s16 = e4m3x2_to_f16x2(static_cast<uint16_t>(scale_row[d / 16])) & 0xFFFFu;
    const uint32_t s2 = s16 | (s16 << 16);
    return make_uint4(hmul2_u32(e2m1x2_byte_to_f16x2<0>(w), s2), hmul2_u32(e2m1x2_byte_to_f16x2<1>(w), s2),
                      hmul2_u32(e2m1x2_byte_to_f16x2<2>(w), s2), hmul2_u32(e2m1x2_byte_to_f16x2<3>(w), s2));
  }
}

// ------------------------------------------------------------------ pass 1
template <int KK, int KV, int D>
__global__ void __launch_bounds__(128) qdequant_kernel(QArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const int p = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  int row, prefix, chunk;
  if (!q_row(a, b, row, prefix, chunk)) return;  // the tensor pass reports it
  const int F = prefix + chunk;
  if (p >= (F + 63) / 64) return;
  int g = a.tables[static_cast<int64_t>(row) * a.L + p];
  if (g < 0 || g >= a.M) {  // never read outside the pool
    if (tid == 0) set_status(a.status, NK_STATUS_PAGE_RANGE);
    g = -1;
  }
  constexpr int KCB = code_row_bytes<KK>(D), VCB = code_row_bytes<KV>(D);
  constexpr int KSB = scale_row_bytes<KK>(D), VSB = scale_row_bytes<KV>(D);
  const int kvalid = g < 0 ? 0 : F - 64 * p;            // rows >= kvalid are stale: zeros
  const int64_t src = g < 0 ? 0 : tile_row(g, h, a.H, a.M, a.head_major);
  const int64_t dst = ((static_cast<int64_t>(b) * a.H + h) * a.L + p) * 64;
  for (int c = tid; c < 64 * (D / 8); c += 128) {
    const int r = c / (D / 8), d = (c % (D / 8)) * 8;
    uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
    if (r < kvalid) {
      kv = dequant8<KK, D>(a.kc + (src + r) * KCB, a.ks + (src + r) * KSB, d);
      vv = dequant8<KV, D>(a.vc + (src + r) * VCB, a.vs + (src + r) * VSB, d);
    }
    *reinterpret_cast<uint4*>(a.scr.k + (dst + r) * D + d) = kv;
    *reinterpret_cast<uint4*>(a.scr.v + (dst + r) * D + d) = vv;
  }
  if (tid < 64) {
    float ksc = 0.f, vsc = 0.f;
    if (tid < kvalid) {
      if constexpr (KK == KIND_FP8) ksc = __half2float(*reinterpret_cast<const __half*>(a.ks + (src + tid) * KSB));
      else if constexpr (KK == KIND_INT8) ksc = ldexpf(1.f, int8_row_shift<D>(a.ks + (src + tid) * KSB));
      else ksc = 1.f;
      if constexpr (KV == KIND_FP8) vsc = __half2float(*reinterpret_cast<const __half*>(a.vs + (src + tid) * VSB));
      else if constexpr (KV == KIND_INT8) vsc = ldexpf(1.f, int8_row_shift<D>(a.vs + (src + tid) * VSB));
      else vsc = 1.f;
    }
    float* sc = a.scr.sc + (dst / 64) * 128;
    sc[tid] = ksc * a.scale_log2;
    sc[64 + tid] = vsc;
  }
}

// ------------------------------------------------------------------ pass 2
template <int D>
struct QCfg {
  static constexpr int THREADS = 192;
  static constexpr int NK = D == 256 ? 3 : 6;
  static constexpr int NV = D == 256 ? 3 : 6;
  static constexpr int KV_BYTES = 64 * D * 2;                 // one f16 page tile
  static constexpr int V_STAGE = KV_BYTES + 1024;             // + the page's 128 scales (512 B)
  static constexpr int OFF_V = NK * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + NV * V_STAGE;
  static constexpr int NBAR = 2 * NK + 2 * NV + 2 + 4;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 64 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0, COL_Q = 128, COL_O = 256;
  static constexpr uint32_t ID_S = tc::idesc_f16(128, 64, false, false);
  static constexpr uint32_t ID_O = tc::idesc_f16(128, D, false, true);
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ void q_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int D>
__global__ void __launch_bounds__(192, 1)
    qprefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, QArgs a) {
  using Cfg = QCfg<D>;
  constexpr int NK = Cfg::NK, NV = Cfg::NV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + Cfg::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;  // [2]
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
  griddep_wait();  // the dequant pass has completed
  griddep_launch_dependents();

  int row, prefix, chunk;
  if (!q_row(a, b, row, prefix, chunk)) {
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
  const int page0 = (b * a.H + h) * a.L + p_lo;  // scratch page of local page 0

  if (tid == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
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
    // -------- TMA producer: f16 K / V tiles and the scales of each page --------
    if (lane == 0) {
      for (int j = 0; j < n; ++j) {
        const int y = (page0 + j) * 64;
        const int ks = j % NK, vs = j % NV;
        if (j >= NK && !mbar_wait_bounded(&k_empty[ks], ((j / NK) - 1) & 1, a.status)) break;
        mbar_arrive_expect_tx(&k_full[ks], Cfg::KV_BYTES);
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb)
          tma_load_2d(sK + ks * Cfg::KV_BYTES + kb * 8192, &tmk, kb * 128, y, &k_full[ks]);
        if (j >= NV && !mbar_wait_bounded(&v_empty[vs], ((j / NV) - 1) & 1, a.status)) break;
        uint8_t* vst = sV + vs * Cfg::V_STAGE;
        mbar_arrive_expect_tx(&v_full[vs], Cfg::KV_BYTES + 512);
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb) tma_load_2d(vst + kb * 8192, &tmv, kb * 128, y, &v_full[vs]);
        bulk_load(vst + Cfg::KV_BYTES, a.scr.sc + static_cast<int64_t>(page0 + j) * 128, 512, &v_full[vs]);
      }
    }
  } else if (warp == 5) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      bool ok = mbar_wait_bounded(q_ready, 0, a.status);
      tc::fence_after();
      for (int j = 0; ok && j <= n; ++j) {
        if (j < n) {
          const int ks = j % NK, sb = j & 1;
          ok = mbar_wait_bounded(&k_full[ks], (j / NK) & 1, a.status);
          if (!ok) break;
          tc::fence_after();
          const uint64_t kd = tc::smem_desc(smem_u32(sK + ks * Cfg::KV_BYTES), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc::mma_ts(tmem + Cfg::COL_S + 64 * sb, tmem + Cfg::COL_Q + kk * 8,
                       kd + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), Cfg::ID_S, kk > 0);
          tc::commit(&s_full[sb]);
          tc::commit(&k_empty[ks]);
        }
        if (j >= 1) {
          const int jj = j - 1, vs = jj % NV;
          ok = mbar_wait_bounded(&v_full[vs], (jj / NV) & 1, a.status);
          if (ok) ok = mbar_wait_bounded(p_full, jj & 1, a.status);
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
      const int e = mx > 0.f ? min(15 - ex, 100) : 0;  // 2^e stays finite in fp32
      const float qf = ldexpf(1.f, e);
      rs = ldexpf(1.f, -e);
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
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) q_arrive(q_ready);
    }
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int sb = j & 1, vs = j % NV;
      ok = mbar_wait_bounded(&s_full[sb], (j / 2) & 1, a.status) && !*s_abort;
      // the page's scales travel with its V tile, which stays until PV(j)
      if (ok) ok = mbar_wait_bounded(&v_full[vs], (j / NV) & 1, a.status) && !*s_abort;
      if (!ok) break;
      tc::fence_after();
      uint32_t v0[32], v1[32];
      tc::ld32(tmem + lane_base + Cfg::COL_S + 64 * sb, v0);
      tc::ld32(tmem + lane_base + Cfg::COL_S + 64 * sb + 32, v1);
      tc::wait_ld();
      const float* ksc = reinterpret_cast<const float*>(sV + vs * Cfg::V_STAGE + Cfg::KV_BYTES);
      const float* vsc = ksc + 64;
      const int kmax = row_valid ? pos - 64 * (p_lo + j) : -1;
      float rmax = -INFINITY;
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 k0 = *reinterpret_cast<const float4*>(ksc + 4 * c4);
        const float4 k1 = *reinterpret_cast<const float4*>(ksc + 32 + 4 * c4);
        const float ka[4] = {k0.x, k0.y, k0.z, k0.w}, kb[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = 4 * c4 + u;
          const float x = c <= kmax ? __uint_as_float(v0[c]) * ka[u] : -INFINITY;
          const float y = 32 + c <= kmax ? __uint_as_float(v1[c]) * kb[u] : -INFINITY;
          v0[c] = __float_as_uint(x);
          v1[c] = __float_as_uint(y);
          rmax = fmaxf(rmax, fmaxf(x, y));
        }
      }
      rmax = rmax == -INFINITY ? -INFINITY : rmax * rs;
      float factor = 1.f;
      const float mnew = fmaxf(m_used, rmax);
      bool resc = false;
      if (mnew != -INFINITY && (m_used == -INFINITY || mnew > m_used + a.thr)) {
        factor = m_used == -INFINITY ? 0.f : ex2(m_used - mnew);
        m_used = mnew;
        resc = true;
      }
      const float mu = m_used == -INFINITY ? 0.f : m_used;
      uint32_t pk[32];
      float sum = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 s0 = *reinterpret_cast<const float4*>(vsc + 4 * c4);
        const float4 s1 = *reinterpret_cast<const float4*>(vsc + 32 + 4 * c4);
        const float sa[4] = {s0.x, s0.y, s0.z, s0.w}, sbv[4] = {s1.x, s1.y, s1.z, s1.w};
        float p0[4], p1[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          p0[u] = ex2(fmaf(__uint_as_float(v0[4 * c4 + u]), rs, -mu));
          p1[u] = ex2(fmaf(__uint_as_float(v1[4 * c4 + u]), rs, -mu));
          sum += p0[u] + p1[u];
        }
        pk[2 * c4] = pack_f16x2(p0[0] * sa[0], p0[1] * sa[1]);
        pk[2 * c4 + 1] = pack_f16x2(p0[2] * sa[2], p0[3] * sa[3]);
        pk[16 + 2 * c4] = pack_f16x2(p1[0] * sbv[0], p1[1] * sbv[1]);
        pk[16 + 2 * c4 + 1] = pack_f16x2(p1[2] * sbv[2], p1[3] * sbv[3]);
      }
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
      prefill_store<D>(tmem + lane_base + Cfg::COL_O, n > 0, row_valid, m_used, l, a.out + orow * D,
                       a.lse ? a.lse + orow : nullptr, a.sp, tile, split, m, s_last);
    }
  }

  if (warp < 4 && tid == 0) mbar_wait_bounded(drain, 0, a.status, 200000000ull);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::dealloc(tmem, Cfg::TMEM_COLS);
}

template <int KK, int KV, int D>
static cudaError_t launch_passes(const CUtensorMap& tk, const CUtensorMap& tv, const QArgs& a, cudaStream_t s) {
  using Cfg = QCfg<D>;
  cudaError_t e = launch_pdl(qdequant_kernel<KK, KV, D>, dim3(a.L, a.H, a.B), dim3(128), 0, s, a);
  if (e != cudaSuccess) return e;
  auto k = qprefill_kernel<D>;
  static bool attr = false;
  if (!attr) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(k, dim3(a.sp.tiles * a.sp.nsplit, a.H, a.B), dim3(Cfg::THREADS), Cfg::SMEM, s, tk, tv, a);
}

template <int KK, int KV>
static cudaError_t launch_qd(int D, const CUtensorMap& tk, const CUtensorMap& tv, const QArgs& a, cudaStream_t s) {
  return D == 256   ? launch_passes<KK, KV, 256>(tk, tv, a, s)
         : D == 128 ? launch_passes<KK, KV, 128>(tk, tv, a, s)
                    : launch_passes<KK, KV, 64>(tk, tv, a, s);
}

size_t qprefill_workspace_bytes(const nk_pool* p, int B) {
  if (p->desc.profile == NK_BF16) return 0;
  return QScratch::bytes(B, p->desc.num_kv_heads, p->L, p->desc.head_dim);
}

// Quantized-pool prefill: dequant pass + tensor pass.  The caller
// (nk_paged_prefill_attention) has checked shapes, pointers and alignment.
int qprefill_launch(const nk_pool* p, int layer, const void* q, const int32_t* tables, const int32_t* table_rows,
                    const int32_t* prefix_len, const int32_t* chunk_len, int B, int Tc, int Hq, float scale_log2,
                    void* out, float* lse, void* ws, size_t ws_bytes, cudaStream_t s) {
  const int D = p->desc.head_dim, H = p->desc.num_kv_heads;
  const int tiles = (Tc + 128 / (Hq / H) - 1) / (128 / (Hq / H));
  const int nsplit = prefill_nsplit(tiles * H * B, p->num_sms);
  const size_t scr = (QScratch::bytes(B, H, p->L, D) + 255) / 256 * 256;
  const size_t need = scr + prefill_split_bytes(B, H, tiles, nsplit, D);
  if (!ws || ws_bytes < need) return fail(NK_ERR_WORKSPACE, "workspace needs " + std::to_string(need) + " bytes");
  if (!aligned16(ws)) return fail(NK_ERR_ALIGN, "workspace must be 16-byte aligned");
  QArgs a;
  const int np = p->n_planes;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.tables = tables;
  a.table_rows = table_rows;
  a.prefix_len = prefix_len;
  a.chunk_len = chunk_len;
  a.kc = static_cast<const uint8_t*>(p->ptrs[layer * np + 0]);
  a.vc = static_cast<const uint8_t*>(p->ptrs[layer * np + 1]);
  a.ks = static_cast<const uint8_t*>(p->ptrs[layer * np + 2]);
  a.vs = static_cast<const uint8_t*>(p->ptrs[layer * np + 3]);
  a.scr = QScratch::at(ws, B, H, p->L, D);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.status = p->status;
  a.scale_log2 = scale_log2;
  a.thr = p->desc.profile == NK_FP8_E4M3_ROW ? 0.f : 8.f;  // FP8-row V carries its scales in P
  a.B = B;
  a.Tc = Tc;
  a.Hq = Hq;
  a.H = H;
  a.G = Hq / H;
  a.L = p->L;
  a.M = p->M;
  a.C = p->desc.max_concurrency;
  a.sp = prefill_split_at(static_cast<char*>(ws) + scr, B, H, tiles, nsplit);
  a.head_major = p->desc.order == NK_HEAD_MAJOR;
  const int64_t rows = static_cast<int64_t>(B) * H * p->L * 64;
  CUtensorMap tk, tv;
  int rc = encode_code_tmap(&tk, a.scr.k, D * 2, rows);
  if (rc) return rc;
  rc = encode_code_tmap(&tv, a.scr.v, D * 2, rows);
  if (rc) return rc;
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
