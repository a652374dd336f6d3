// prefill.cu -- chunked prefill / replay attention through the block tables on
// the 5th-generation tensor cores (tcgen05, operands and accumulators in TMEM).
//
// Contract: query i < chunk_len[b] of row b sits at logical position
// prefix_len[b] + i and attends keys j <= prefix_len[b] + i of its table row
// ("Paged KV cache" maintainer design page: pages are read in place through
// the block table, a frontier may sit mid-page); the work is proportional to
// the query-key pairs prefix * S + S (S + 1) / 2 ("Resource scheduling and
// context cache" page, machine cost model).  BF16 pools.
//
// Tile.  A CTA owns 128 query rows of one (row b, KV head h): TQ = 128 / G
// consecutive chunk tokens times the G query heads that share KV head h, so
// every K / V page tile is loaded once for all of them.  Keys advance one page
// (64 keys) at a time, which is also the P = 64 pipeline unit:
//   S   = Q K^T   tcgen05.mma, M 128 x N 64 x K D, A = Q (TMEM, written once
//                 by the softmax warps), B = K page tile (shared, K-major,
//                 128-byte swizzle), fp32 accumulator in TMEM (two buffers);
//   P   = exp2(S * scale * log2 e - m) in bf16, written by the four softmax
//                 warps (one TMEM lane = one query row each) over the first
//                 32 columns of the S buffer it was computed from;
//   O  += P V     tcgen05.mma, M 128 x N D x K 64, A = P (TMEM), B = V page
//                 tile (shared, MN-major), fp32 accumulator in TMEM.
// With both A operands in TMEM, the only shared-memory operand traffic is the
// K and V page tiles.  The MMAs of one thread execute in issue order, so the
// next S into a buffer (issued after the PV that reads its P) cannot overwrite
// P early.  The running max is rescaled lazily: O is rescaled only when the
// row max grows by more than 2^8, so P stays below 256 and fp32 O never
// overflows.
//
// TMEM columns: S buffers [0, 64) and [64, 128), Q [128, 128 + D/2),
// O [256, 256 + D).
//
// Warp roles (192 threads): warps 0-3 softmax and epilogue (and the Q copy to
// TMEM), warp 4 TMA producer (K and V page tiles through two rings), warp 5 the
// single MMA-issuing thread.  All waits are bounded.
#include <cmath>

#include "internal.h"
#include "prefill_split.cuh"
#include "tcgen05.cuh"

namespace nk {

struct PrefillArgs {
  const __nv_bfloat16* q;  // [B][Tc][Hq][D]
  const int32_t* tables;
  const int32_t* table_rows;
  const int32_t* prefix_len;
  const int32_t* chunk_len;
  __nv_bfloat16* out;
  float* lse;
  int* status;
  float scale_log2;  // softmax_scale * log2(e)
  int B, Tc, Hq, H, G, L, M, C;
  PrefillSplit sp;
  int head_major;  // plane order
};

template <int D>
struct PrefillCfg {
  static constexpr int THREADS = 192;
  static constexpr int NK = D == 256 ? 3 : 6;  // K ring
  static constexpr int NV = D == 256 ? 3 : 6;  // V ring
  static constexpr int KV_BYTES = 64 * D * 2;  // one page tile, D/64 column blocks of 8 KB
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + NV * KV_BYTES;
  static constexpr int NBAR = 2 * NK + 2 * NV + 2 + 4;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 64 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0, COL_Q = 128, COL_O = 256;
  static constexpr uint32_t ID_S = tc::idesc_bf16(128, 64, false, false);
  static constexpr uint32_t ID_O = tc::idesc_bf16(128, D, false, true);
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ void arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int D>
__global__ void __launch_bounds__(192, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   PrefillArgs a) {
  using Cfg = PrefillCfg<D>;
  constexpr int NK = Cfg::NK, NV = Cfg::NV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + Cfg::OFF_K;
  uint8_t* sV = smem + Cfg::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;   // [2]
  uint64_t* p_full = s_full + 2;     // [1]
  uint64_t* o_done = p_full + 1;     // [1]
  uint64_t* q_ready = o_done + 1;    // [1]
  uint64_t* drain = q_ready + 1;     // [1]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* s_last = s_abort + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x / a.sp.nsplit, split = blockIdx.x % a.sp.nsplit;
  const int h = blockIdx.y, b = blockIdx.z;
  const int G = a.G, TQ = 128 / G;
  griddep_wait();  // launched with programmatic stream serialization
  griddep_launch_dependents();

  // ---- row geometry (uniform across the CTA) -------------------------------
  const int row = a.table_rows[b];
  int prefix = a.prefix_len[b], chunk = a.chunk_len[b];
  if (row < 0 || row >= a.C || prefix < 0 || chunk < 0 || chunk > a.Tc ||
      static_cast<int64_t>(prefix) + chunk > static_cast<int64_t>(a.L) * 64) {
    if (tid == 0 && qt == 0 && h == 0) set_status(a.status, NK_STATUS_FRONTIER);
    return;
  }
  const int t0 = qt * TQ;
  if (t0 >= chunk) return;  // no query of this tile is in the chunk
  const int t_last = min(t0 + TQ, chunk) - 1;
  const int nkt = (prefix + t_last + 1 + 63) / 64;  // key pages of the tile
  // this split's pages [p_lo, p_lo + n); local page i is absolute page p_lo + i
  const int per = (nkt + a.sp.nsplit - 1) / a.sp.nsplit;
  const int p_lo = min(split * per, nkt);
  const int n = min(p_lo + per, nkt) - p_lo;
  const int32_t* table = a.tables + static_cast<int64_t>(row) * a.L + p_lo;

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
    // ------------------------------ TMA producer ------------------------------
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
        const int ks = j % NK, vs = j % NV;
        if (j >= NK && !mbar_wait_bounded(&k_empty[ks], ((j / NK) - 1) & 1, a.status)) stop = 1;
        if (!stop) {
          mbar_arrive_expect_tx(&k_full[ks], Cfg::KV_BYTES);
#pragma unroll
          for (int kb = 0; kb < D / 64; ++kb)
            tma_load_2d(sK + ks * Cfg::KV_BYTES + kb * 8192, &tmk, kb * 128, y, &k_full[ks]);
        }
        if (!stop && j >= NV && !mbar_wait_bounded(&v_empty[vs], ((j / NV) - 1) & 1, a.status)) stop = 1;
        if (!stop) {
          mbar_arrive_expect_tx(&v_full[vs], Cfg::KV_BYTES);
#pragma unroll
          for (int kb = 0; kb < D / 64; ++kb)
            tma_load_2d(sV + vs * Cfg::KV_BYTES + kb * 8192, &tmv, kb * 128, y, &v_full[vs]);
        }
        if (stop) *s_abort = 1;
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) break;
    }
  } else if (warp == 5) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      bool ok = mbar_wait_bounded(q_ready, 0, a.status);
      tc::fence_after();
      for (int j = 0; ok && j <= n; ++j) {
        if (j < n) {  // S(j) = Q K(j)^T into buffer j & 1
          const int ks = j % NK, sb = j & 1;
          ok = mbar_wait_bounded(&k_full[ks], (j / NK) & 1, a.status);
          if (!ok) break;
          tc::fence_after();
          const uint64_t kd = tc::smem_desc(smem_u32(sK + ks * Cfg::KV_BYTES), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)  // 16 dims: 8 TMEM columns of Q, 32 bytes of a K row
            tc::mma_ts(tmem + Cfg::COL_S + 64 * sb, tmem + Cfg::COL_Q + kk * 8,
                       kd + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), Cfg::ID_S, kk > 0);
          tc::commit(&s_full[sb]);
          tc::commit(&k_empty[ks]);
        }
        if (j >= 1) {  // O += P(j - 1) V(j - 1), P in the first 32 columns of buffer (j - 1) & 1
          const int jj = j - 1, vs = jj % NV;
          ok = mbar_wait_bounded(&v_full[vs], (jj / NV) & 1, a.status);
          if (ok) ok = mbar_wait_bounded(p_full, jj & 1, a.status);
          if (!ok) break;
          tc::fence_after();
          const uint64_t vd = tc::smem_desc(smem_u32(sV + vs * Cfg::KV_BYTES), 8192, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // 16 keys: 8 TMEM columns of P, 2 KB of V rows
            tc::mma_ts(tmem + Cfg::COL_O, tmem + Cfg::COL_S + 64 * (jj & 1) + kk * 8,
                       vd + static_cast<uint64_t>((kk * 2048) >> 4), Cfg::ID_O, (jj > 0 || kk > 0));
          tc::commit(o_done);
          tc::commit(&v_empty[vs]);
        }
      }
      if (!ok) *s_abort = 1;
      tc::commit(drain);  // arrives once every MMA issued above has completed
    }
  } else {
    // ------------------------------ softmax warps -----------------------------
    const int m = tid;  // query row = TMEM lane
    const int tl = m / G, g = m % G;
    const int token = t0 + tl;
    const bool row_valid = token < chunk;
    const int pos = prefix + token;  // keys <= pos are visible
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // Q row m to TMEM columns [COL_Q, COL_Q + D/2): column c holds dims 2c, 2c+1
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + ((static_cast<int64_t>(b) * a.Tc + token) * a.Hq + h * G + g) * D);
#pragma unroll 1
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t qv[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = row_valid ? src[c0 / 4 + u] : make_uint4(0u, 0u, 0u, 0u);
          qv[4 * u] = x.x;
          qv[4 * u + 1] = x.y;
          qv[4 * u + 2] = x.z;
          qv[4 * u + 3] = x.w;
        }
        tc::st32(tmem + lane_base + Cfg::COL_Q + c0, qv);
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) arrive(q_ready);
    }
    float m_used = -INFINITY, l = 0.f;
    const bool pos_scale = a.scale_log2 >= 0.f;
    const float fill = pos_scale ? -INFINITY : INFINITY;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int sb = j & 1;
      ok = mbar_wait_bounded(&s_full[sb], (j / 2) & 1, a.status) && !*s_abort;
      if (!ok) break;
      tc::fence_after();
      uint32_t v0[32], v1[32];
      tc::ld32(tmem + lane_base + Cfg::COL_S + 64 * sb, v0);
      tc::ld32(tmem + lane_base + Cfg::COL_S + 64 * sb + 32, v1);
      tc::wait_ld();
      // The row maximum of the scaled scores is the scale times the largest
      // raw score (the smallest one for a negative scale); masked keys get the
      // fill value that no extremum picks and whose exponent is 0.  The causal
      // mask is applied only where the page reaches past a row's last key.
      const int kmax = row_valid ? pos - 64 * (p_lo + j) : -1;  // keys c <= kmax of this page are visible
      float rext = fill;
      if (__all_sync(0xffffffffu, kmax >= 63)) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float x = __uint_as_float(v0[c]), y = __uint_as_float(v1[c]);
          rext = pos_scale ? fmaxf(rext, fmaxf(x, y)) : fminf(rext, fminf(x, y));
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c > kmax) v0[c] = __float_as_uint(fill);
          if (32 + c > kmax) v1[c] = __float_as_uint(fill);
          const float x = __uint_as_float(v0[c]), y = __uint_as_float(v1[c]);
          rext = pos_scale ? fmaxf(rext, fmaxf(x, y)) : fminf(rext, fminf(x, y));
        }
      }
      const float rmax = rext == fill ? -INFINITY : rext * a.scale_log2;
      float factor = 1.f;
      const float mnew = fmaxf(m_used, rmax);
      bool resc = false;
      if (mnew != -INFINITY && (m_used == -INFINITY || mnew > m_used + 8.f)) {
        factor = m_used == -INFINITY ? 0.f : ex2(m_used - mnew);
        m_used = mnew;
        resc = true;
      }
      const float mu = m_used == -INFINITY ? 0.f : m_used;
      uint32_t pk[32];
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float pa = ex2(fmaf(__uint_as_float(v0[2 * c]), a.scale_log2, -mu));
        const float pb = ex2(fmaf(__uint_as_float(v0[2 * c + 1]), a.scale_log2, -mu));
        const float pc = ex2(fmaf(__uint_as_float(v1[2 * c]), a.scale_log2, -mu));
        const float pd = ex2(fmaf(__uint_as_float(v1[2 * c + 1]), a.scale_log2, -mu));
        sum += (pa + pb) + (pc + pd);
        pk[c] = pack_bf16x2(pa, pb);
        pk[16 + c] = pack_bf16x2(pc, pd);
      }
      l = l * factor + sum;
      // Consume PV(j - 1)'s completion every page (an mbarrier parity wait is
      // only sound one phase at a time); it is normally done by now, and O
      // must be complete before a rescale.
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
      // P over the first 32 columns of this S buffer (this warp has read them)
      tc::st32(tmem + lane_base + Cfg::COL_S + 64 * sb, pk);
      tc::wait_st();
      // Rows of the V page past the row's frontier hold stale bytes (possibly
      // NaN); their P is 0, but 0 * NaN would still poison O, so zero them.
      const int kstale = prefix + chunk - 64 * (p_lo + j);
      if (kstale < 64) {
        const int vs = j % NV;
        ok = mbar_wait_bounded(&v_full[vs], (j / NV) & 1, a.status);
        uint8_t* vt = sV + vs * Cfg::KV_BYTES;
        const int nrow = 64 - kstale;
        for (int i2 = tid; i2 < nrow * (D / 64) * 8; i2 += 128) {
          const int rr = kstale + i2 / ((D / 64) * 8), rem = i2 % ((D / 64) * 8);
          *reinterpret_cast<uint4*>(vt + (rem >> 3) * 8192 + rr * 128 + (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (!ok) break;
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) arrive(p_full);
    }
    // ---- epilogue: O / l to bf16, or this split's partial and the merge ------
    if (ok && n > 0) ok = mbar_wait_bounded(o_done, (n - 1) & 1, a.status) && !*s_abort;
    tc::fence_after();
    if (ok) {
      const int64_t orow = (static_cast<int64_t>(b) * a.Tc + token) * a.Hq + h * G + g;
      const int64_t tile = (static_cast<int64_t>(b) * a.H + h) * a.sp.tiles + qt;
      prefill_store<D>(tmem + lane_base + Cfg::COL_O, n > 0, row_valid, m_used, l, a.out + orow * D,
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

template <int D>
static cudaError_t launch_prefill(const nk_pool* p, int layer, const PrefillArgs& a, dim3 grid, cudaStream_t s) {
  using Cfg = PrefillCfg<D>;
  auto k = prefill_kernel<D>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(k, grid, dim3(Cfg::THREADS), Cfg::SMEM, s, p->tmap[layer * 2 + 0], p->tmap[layer * 2 + 1], a);
}

}  // namespace nk

namespace nk {
int qprefill_launch(const nk_pool* p, int layer, const void* q, const int32_t* tables, const int32_t* table_rows,
                    const int32_t* prefix_len, const int32_t* chunk_len, int B, int Tc, int Hq, float scale_log2,
                    void* out, float* lse, void* ws, size_t ws_bytes, cudaStream_t s);
}  // namespace nk

using namespace nk;

extern "C" int nk_prefill_workspace_bytes(const nk_pool* pool, int32_t B, int32_t Tc, int32_t Hq,
                                          size_t* bytes) {
  clear_error();
  if (!pool || !bytes) return fail(NK_ERR_INVALID_ARG, "null argument");
  if (Hq < 1 || Hq % pool->desc.num_kv_heads || Tc < 1 || B < 1) return fail(NK_ERR_SHAPE, "bad B, Tc or Hq");
  // every profile: when the tiles are split over their pages, the partials
  // and counters (zero-filled before the first use, left at zero by every
  // call); the size depends on B, H, Tc and D, never on the context
  const int H = pool->desc.num_kv_heads, G = Hq / H;
  if (G > 16 || 128 % G) return fail(NK_ERR_UNSUPPORTED, "GQA group must divide 128 and be <= 16");
  const int tiles = (Tc + 128 / G - 1) / (128 / G);
  const int nsplit = prefill_nsplit(tiles * H * B, pool->num_sms);
  *bytes = prefill_split_bytes(B, H, tiles, nsplit, pool->desc.head_dim);
  return NK_OK;
}

extern "C" int nk_paged_prefill_attention(const void* q_chunk, int32_t Hq, const nk_pool* pool,
                                          int32_t layer, const int32_t* block_tables,
                                          const int32_t* table_rows, const int32_t* prefix_len,
                                          const int32_t* chunk_len, int32_t B, int32_t Tc,
                                          float softmax_scale, void* out, float* lse,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  if (!q_chunk || !pool || !block_tables || !table_rows || !prefix_len || !chunk_len || !out)
    return fail(NK_ERR_INVALID_ARG, "null argument to nk_paged_prefill_attention");
  if (!std::isfinite(softmax_scale)) return fail(NK_ERR_INVALID_ARG, "softmax_scale is not finite");
  const int D = pool->desc.head_dim, H = pool->desc.num_kv_heads;
  if (D != 64 && D != 128 && D != 256) return fail(NK_ERR_UNSUPPORTED, "chunked prefill needs head_dim 64, 128 or 256");
  if (layer < 0 || layer >= pool->desc.num_layers) return fail(NK_ERR_SHAPE, "layer out of range");
  if (B < 1 || B > pool->desc.max_concurrency) return fail(NK_ERR_SHAPE, "B must be in [1, C]");
  if (Tc < 1) return fail(NK_ERR_SHAPE, "Tc must be >= 1");
  if (Hq < 1 || Hq % H) return fail(NK_ERR_SHAPE, "Hq must be a positive multiple of num_kv_heads");
  const int G = Hq / H;
  if (G > 16 || 128 % G) return fail(NK_ERR_UNSUPPORTED, "GQA group must divide 128 and be <= 16");
  if (!aligned16(q_chunk) || !aligned16(out)) return fail(NK_ERR_ALIGN, "q / out must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pool->desc.profile != NK_BF16)
    return qprefill_launch(pool, layer, q_chunk, block_tables, table_rows, prefix_len, chunk_len, B, Tc, Hq,
                           softmax_scale * 1.4426950408889634f, out, lse, workspace, workspace_bytes, s);
  PrefillArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q_chunk);
  a.tables = block_tables;
  a.table_rows = table_rows;
  a.prefix_len = prefix_len;
  a.chunk_len = chunk_len;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.status = pool->status;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.B = B;
  a.Tc = Tc;
  a.Hq = Hq;
  a.H = H;
  a.G = G;
  a.L = pool->L;
  a.M = pool->M;
  a.C = pool->desc.max_concurrency;
  a.head_major = pool->desc.order == NK_HEAD_MAJOR;
  const int TQ = 128 / G;
  const int tiles = (Tc + TQ - 1) / TQ;
  const int nsplit = prefill_nsplit(tiles * H * B, pool->num_sms);
  const size_t need = prefill_split_bytes(B, H, tiles, nsplit, D);
  if (need && (!workspace || workspace_bytes < need))
    return fail(NK_ERR_WORKSPACE, "workspace needs " + std::to_string(need) + " bytes");
  if (need && !aligned16(workspace)) return fail(NK_ERR_ALIGN, "workspace must be 16-byte aligned");
  a.sp = prefill_split_at(workspace, B, H, tiles, nsplit);
  const dim3 grid(tiles * nsplit, H, B);
  cudaError_t e = D == 256   ? launch_prefill<256>(pool, layer, a, grid, s)
                  : D == 128 ? launch_prefill<128>(pool, layer, a, grid, s)
                             : launch_prefill<64>(pool, layer, a, grid, s);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return NK_OK;
}
