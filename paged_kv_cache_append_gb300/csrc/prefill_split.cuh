// prefill_split.cuh -- the output stage shared by the tcgen05 prefill kernels
// (prefill.cu, qprefill.cu), with an optional split of each tile's key pages.
//
// A tile is 128 query rows of one (row b, KV head h).  With nsplit > 1 the
// tile's pages are cut into nsplit contiguous ranges, one CTA each, so that a
// launch of T tiles runs as T * nsplit CTAs and its last wave of 1-CTA-per-SM
// work is fuller.  Every split writes its partial (m, l, O) for the 128 rows
// -- O unnormalised, relative to 2^m -- to the workspace, then counts itself
// on the tile's counter; the split that brings the counter to nsplit merges
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  out = sum_s O_s 2^(m_s - M) / L,
//   lse = (M + log2 L) ln 2
// (the softmax over the union of the ranges) and resets the counter.  A split
// with no page (a short tile) contributes l = 0 and no O.
#pragma once

#include "device.cuh"
#include "tcgen05.cuh"

namespace nk {

struct PrefillSplit {
  int nsplit;      // splits per tile (1: no partials)
  int tiles;       // tiles per (row, KV head)
  int* counters;   // [B][H][tiles], zero between calls
  float2* ws_ml;   // [B][H][tiles][nsplit][128] (m, l)
  float* ws_o;     // [B][H][tiles][nsplit][128][D]
};

// Layout of the split workspace after `base` bytes of other scratch.
__host__ __device__ inline size_t prefill_split_bytes(int B, int H, int tiles, int nsplit, int D) {
  if (nsplit <= 1) return 0;
  const size_t t = static_cast<size_t>(B) * H * tiles;
  const size_t cnt = (t * 4 + 255) / 256 * 256;
  const size_t ml = (t * nsplit * 128 * 8 + 255) / 256 * 256;
  return cnt + ml + t * nsplit * 128 * static_cast<size_t>(D) * 4;
}

inline PrefillSplit prefill_split_at(void* ws, int B, int H, int tiles, int nsplit) {
  PrefillSplit sp{nsplit, tiles, nullptr, nullptr, nullptr};
  if (nsplit <= 1) return sp;
  const size_t t = static_cast<size_t>(B) * H * tiles;
  const size_t cnt = (t * 4 + 255) / 256 * 256;
  const size_t ml = (t * nsplit * 128 * 8 + 255) / 256 * 256;
  char* p = static_cast<char*>(ws);
  sp.counters = reinterpret_cast<int*>(p);
  sp.ws_ml = reinterpret_cast<float2*>(p + cnt);
  sp.ws_o = reinterpret_cast<float*>(p + cnt + ml);
  return sp;
}

// Splits per tile: the smallest of 1..4 that minimises the waves of
// 1-CTA-per-SM work per unit of work (ceil(ctas / sms) / nsplit).
inline int prefill_nsplit(int ctas, int sms) {
  int best = 1;
  double best_w = 1e30;
  for (int s = 1; s <= 4; ++s) {
    const double w = static_cast<double>((ctas * s + sms - 1) / sms) / s;
    if (w < best_w - 1e-9) {
      best_w = w;
      best = s;
    }
  }
  return best;
}

// Output of one softmax thread (query row m of the tile).  has_o: the split
// visited at least one page (TMEM O is valid).  Called by the 128 softmax
// threads together (named barrier 1).
template <int D>
__device__ __forceinline__ void prefill_store(uint32_t tmem_o, bool has_o, bool row_valid, float m_used, float l,
                                              __nv_bfloat16* out_row, float* lse_at, const PrefillSplit& sp,
                                              int64_t tile, int split, int m, volatile int* s_last) {
  if (sp.nsplit <= 1) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t ov[32];
      if (has_o) {
        tc::ld32(tmem_o + c0, ov);
        tc::wait_ld();
      }
      if (row_valid) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = has_o ? pack_bf16x2(__uint_as_float(ov[2 * c]) * inv, __uint_as_float(ov[2 * c + 1]) * inv) : 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(out_row + c0 + 8 * c) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
    }
    if (row_valid && lse_at) *lse_at = l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
    return;
  }
  // ---- partial of this split ------------------------------------------------
  const int64_t part = tile * sp.nsplit + split;
  float* po = sp.ws_o + (part * 128 + m) * D;
  sp.ws_ml[part * 128 + m] = make_float2(has_o ? m_used : -INFINITY, has_o ? l : 0.f);
  if (has_o) {
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t ov[32];
      tc::ld32(tmem_o + c0, ov);
      tc::wait_ld();
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(po + c0 + 4 * c) = make_uint4(ov[4 * c], ov[4 * c + 1], ov[4 * c + 2], ov[4 * c + 3]);
    }
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
  if (m == 0) {
    __threadfence();
    const int done = atomicAdd(&sp.counters[tile], 1);
    *s_last = (done == sp.nsplit - 1);
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
  if (!*s_last) return;
  __threadfence();
  // ---- merge (last split of the tile) ------------------------------------------
  const int64_t p0 = tile * sp.nsplit;
  float M = -INFINITY;
  for (int s = 0; s < sp.nsplit; ++s) M = fmaxf(M, __ldcg(&sp.ws_ml[(p0 + s) * 128 + m]).x);
  float L = 0.f;
  for (int s = 0; s < sp.nsplit; ++s) {
    const float2 ml = __ldcg(&sp.ws_ml[(p0 + s) * 128 + m]);
    if (ml.y > 0.f) L += ml.y * ex2(ml.x - M);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    float acc[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) acc[c] = 0.f;
    for (int s = 0; s < sp.nsplit; ++s) {
      const float2 ml = __ldcg(&sp.ws_ml[(p0 + s) * 128 + m]);
      if (!(ml.y > 0.f)) continue;  // an empty split has no O
      const float w = ex2(ml.x - M) * inv;
      const float4* src = reinterpret_cast<const float4*>(sp.ws_o + ((p0 + s) * 128 + m) * D + c0);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 v = __ldcg(src + c);
        acc[4 * c] = fmaf(w, v.x, acc[4 * c]);
        acc[4 * c + 1] = fmaf(w, v.y, acc[4 * c + 1]);
        acc[4 * c + 2] = fmaf(w, v.z, acc[4 * c + 2]);
        acc[4 * c + 3] = fmaf(w, v.w, acc[4 * c + 3]);
      }
    }
    if (row_valid) {
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(acc[2 * c], acc[2 * c + 1]);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(out_row + c0 + 8 * c) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    }
  }
  if (row_valid && lse_at) *lse_at = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  if (m == 0) sp.counters[tile] = 0;  // ready for the next call
}

}  // namespace nk
