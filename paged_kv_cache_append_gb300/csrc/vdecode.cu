// vdecode.cu -- decode / verify attention for 17..32 query rows per KV head
// (T * G > 16, e.g. a 4-token verify with a GQA group of 8) over FP8-row,
// NVFP4-G16 and K8V4 pools, on the 5th-generation tensor cores.
//
// Same contract, split plan, workspace layout and merge as the warp-level
// decode (decode.cuh): a CTA owns one (row b, KV head h, page range) and
// writes the final out / lse when its row has one split, else a partial
// (m, l, acc) that merge_kernel combines.  With 32 query rows the warp-level
// kernel keeps 128 fp32 accumulators per thread in registers and is bound by
// its mma.sync issue rate; here S and O live in tensor memory.  Two forms:
//
//   vtdecode_kernel (head_dim 64, 128): S^T = K Q^T and O^T = V^T P^T, the
//     tile's 128 keys as M and the 32 query rows as N; the keys are
//     dequantized straight into TMEM (the A operand of S^T).  Described
//     above the kernel.
//   vdecode_kernel (head_dim 256): S = Q K^T and O += P V with the query
//     rows in TMEM lanes and the f16 K tile in shared memory, as below.
//
// vdecode_kernel: a key tile is TK = 64 keys (one page) at head_dim 256,
// 128 keys (two pages) at smaller head_dims:
//   S = Q K^T   tcgen05.mma M 128 x N TK x K D; Q (f16, each query row scaled
//               by a power of two) in TMEM, K = the tile dequantized to f16 in
//               shared memory;
//   O += P V    tcgen05.mma M 128 x N D x K TK; P (f16) over its S buffer.
// Operands are exact: E4M3 and E2M1 codes are f16 values, an E2M1 code times
// its E4M3 scale is an exact f16 product, FP8-row key scales multiply the fp32
// scores and FP8-row value scales the softmax weights.  Rows rescale lazily
// (p <= 2^8); FP8-row weights p * s are lifted by 2^K (v_lift), so that they
// stay finite and clear of f16's subnormal range for V of any magnitude.
//
// Layout of the query rows.  Query row r sits in TMEM lane 32 (r / 8) + r % 8,
// so that each of the four lane quadrants (and each warp scheduler) holds 8
// rows; the other 24 lanes of a quadrant carry zero rows of Q.  A softmax warp
// per quadrant reads S with the 16x256b shape (4 threads per row) and writes P
// back in the same shape, which puts the keys of P in a fixed order inside
// every 16-key group; the dequantizing warps store the V tile's rows in that
// order (vrow), so P V sums over matching keys.
//
// Warps of both kernels (448 threads): 0-3 softmax and output (one per lane
// quadrant), 4-11 dequantize tiles (and, in the fused call, encode the new
// tokens first), 12 is the TMA producer of raw code / scale pages, 13 issues
// the MMAs.  All waits are bounded.
#include "decode.cuh"
#include "tcgen05.cuh"

namespace nk {

template <int KK, int KV, int D>
struct VCfg {
  static constexpr int THREADS = 448, NDW = 8;  // threads; dequantizing warps
  static constexpr int TK = D <= 128 ? 128 : 64, PPT = TK / 64;  // keys and pages of a tile
  // 8-code units: thread dt of the dequantizing warps converts column unit
  // p = dt % (D / 8) of rows r0 + RPT k, r0 = dt / (D / 8), of every page
  static constexpr int RPT = 2048 / D, PASSES = 64 / RPT;
  static constexpr int KCB = code_row_bytes<KK>(D), VCB = code_row_bytes<KV>(D);
  static constexpr int KSB = scale_row_bytes<KK>(D), VSB = scale_row_bytes<KV>(D);
  static constexpr int K_RB = KCB < 128 ? KCB : 128, V_RB = VCB < 128 ? VCB : 128;
  static constexpr int R_KS = align_up(64 * KCB, 1024);             // raw page stage: K codes, V codes,
  static constexpr int R_KSC = R_KS + align_up(64 * VCB, 1024);     // K scales, V scales
  static constexpr int R_VSC = R_KSC + align_up(64 * KSB, 128);
  static constexpr int RAW = align_up(R_VSC + 64 * VSB, 1024);
  static constexpr int TX = 64 * (KCB + VCB + KSB + VSB);
  static constexpr int F16 = TK * D * 2;       // f16 tile: D / 64 chunks of TK rows x 128 bytes
  static constexpr int CHUNK = TK * 128;
  static constexpr int NK = 2, NV = 2, NS = 4;
  static constexpr int NSB = 2;                // S buffers in TMEM (P is written over its S)
  // raw page stages: as many as fit next to the f16 tiles
  static constexpr int NR_FIT = (204 * 1024 - (NK + NV) * F16 - 6144) / RAW;
  static constexpr int NR = NR_FIT < 2 * PPT ? 2 * PPT : NR_FIT > 8 ? 8 : NR_FIT;
  static constexpr int OFF_KF = NR * RAW;
  static constexpr int OFF_VF = OFF_KF + NK * F16;
  static constexpr int OFF_SC = OFF_VF + NV * F16;   // [NS][2 TK] float: key factors, value scales
  static constexpr int OFF_BAR = OFF_SC + NS * 2 * TK * 4;
  static constexpr int NBAR = 2 * NR + 2 * NK + 2 * NV + NS + 3 * NSB + 3;
  // at least half of the SM's shared memory: one CTA per SM owns all 512 TMEM columns
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 128 + 1024;
  static constexpr int SMEM = SMEM_USED > 116 * 1024 ? SMEM_USED : 116 * 1024;
  // TMEM columns: S buffers from 0, the O accumulator at 256, Q in the gap
  // below 256 when it fits there, else right after O
  static constexpr uint32_t COL_S = 0, COL_O = 256;
  static constexpr uint32_t COL_Q = TK * NSB + D / 2 <= 256 ? TK * NSB : 256 + D;
  static_assert(COL_O + D <= 512 && COL_Q + D / 2 <= 512 && TK * NSB <= 256, "TMEM columns");
  static constexpr uint32_t ID_S = tc::idesc_f16(128, TK, false, false);
  static constexpr uint32_t ID_O = tc::idesc_f16(128, D, false, true);
  static constexpr float THR = 8.f;  // lazy rescale threshold (log2 units): p <= 2^8
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
  static_assert(RPT * (D / 8) == 32 * NDW && PASSES * RPT == 64 && RPT % 8 == 0, "unit map");
};

// Four E4M3 codes -> two f16x2 (exact).
__device__ __forceinline__ void e4m3x4_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Eight E2M1 codes (low nibble first) -> four f16x2 (exact).
__device__ __forceinline__ void e2m1x8_f16(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2, uint32_t& h3) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}

// Row of the V tile that holds key r of the page: inside each 16-key group,
// key bits (b3 b2 b1 b0) go to row bits (b2 b1 b3 b0), the order in which the
// softmax warps' 16x256b stores lay out P.
__device__ __forceinline__ int vrow(int r) { return (r & ~15) | ((r & 6) << 1) | ((r & 8) >> 2) | (r & 1); }

// One 8-code unit: dims [8 p, 8 p + 8) of one key.  The raw bytes of all of
// a thread's units are loaded first (RawUnit), then converted to 8 exact f16
// values each and stored, so that the shared-memory loads are not ordered
// behind the stores of earlier units.
struct RawUnit {
  uint32_t w0, w1, s;  // FP8: 8 codes in w0, w1; NVFP4: 8 codes in w0 and the E4M3 scale byte in s
};

template <int KIND>
__device__ __forceinline__ RawUnit ld_unit(const uint8_t* src, const uint8_t* sc) {
  RawUnit u;
  if constexpr (KIND == KIND_FP8) {
    const uint2 w = *reinterpret_cast<const uint2*>(src);
    u.w0 = w.x;
    u.w1 = w.y;
    u.s = 0u;
  } else {
    u.w0 = *reinterpret_cast<const uint32_t*>(src);
    u.w1 = 0u;
    u.s = *sc;
  }
  return u;
}

// Converts a unit and stores its 16 bytes of f16; zero when the key lies past
// the frontier or the tile's pages.
template <int KIND>
__device__ __forceinline__ void cvt_unit(const RawUnit& u, uint8_t* dst, bool zero) {
  uint32_t h[4];
  if (zero) {
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = 0u;
  } else if constexpr (KIND == KIND_FP8) {
    e4m3x4_f16(u.w0, h[0], h[1]);
    e4m3x4_f16(u.w1, h[2], h[3]);
  } else {
    const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint16_t>(u.s * 0x101u));  // the scale in both halves
    e2m1x8_f16(u.w0, h[0], h[1], h[2], h[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = hmul2_u32(h[i], s2);
  }
  *reinterpret_cast<uint4*>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
}

// Byte offsets of a thread's first unit (row r0, column unit p) in a raw page
// stage and in the f16 tile (row `frow` of the tile); the other units of the
// thread follow at fixed strides, as RPT is a multiple of 8 (the swizzle
// phase of the row does not change).
template <int KIND, int D>
__device__ __forceinline__ int raw_off(int r0, int p) {
  constexpr int CB = code_row_bytes<KIND>(D), RB = CB < 128 ? CB : 128;
  const int col = KIND == KIND_FP8 ? 8 * p : 4 * p;
  return (col / RB) * (64 * RB) + static_cast<int>(swz<RB>(r0, col % RB));
}

template <int TK>
__device__ __forceinline__ int f16_off(int frow, int p) {
  return (p / 8) * (TK * 128) + static_cast<int>(swz<128>(frow, (p % 8) * 16));
}

__device__ __forceinline__ void v_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int KK, int KV, int D>
__global__ void __launch_bounds__(448, 1)
    vdecode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, DecodeArgs a) {
  using Cfg = VCfg<KK, KV, D>;
  constexpr int NR = Cfg::NR, NK = Cfg::NK, NV = Cfg::NV, NS = Cfg::NS, NDW = Cfg::NDW, NSB = Cfg::NSB;
  constexpr int TK = Cfg::TK, PPT = Cfg::PPT;
  constexpr int R = 32;  // query rows of a part in the workspace
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKf = smem + Cfg::OFF_KF;
  uint8_t* sVf = smem + Cfg::OFF_VF;
  float* sSc = reinterpret_cast<float*>(smem + Cfg::OFF_SC);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* raw_full = bars;             // [NR] raw page stages
  uint64_t* raw_empty = raw_full + NR;
  uint64_t* kf_full = raw_empty + NR;    // [NK] f16 K tiles
  uint64_t* kf_empty = kf_full + NK;
  uint64_t* vf_full = kf_empty + NK;     // [NV] f16 V tiles
  uint64_t* vf_empty = vf_full + NV;
  uint64_t* sc_full = vf_empty + NV;     // [NS] key factors / value scales of a tile
  uint64_t* s_full = sc_full + NS;       // [NSB]: S(j) in buffer j % NSB
  uint64_t* p_full = s_full + NSB;       // [NSB]: P(j) written over it
  uint64_t* o_done = p_full + NSB;       // [NSB]: P V(j) accumulated
  uint64_t* q_ready = o_done + NSB;
  uint64_t* app = q_ready + 1;
  uint64_t* drain = app + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
  int* s_F = reinterpret_cast<int*>(tslot + 2);     // [8]
  int* s_row = s_F + 8;                             // [8]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  if (tid == 0) {
    for (int i = 0; i < NR; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], NDW);
    }
    for (int i = 0; i < NK; ++i) {
      mbar_init(&kf_full[i], NDW);
      mbar_init(&kf_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&vf_full[i], NDW);
      mbar_init(&vf_empty[i], 1);
    }
    for (int i = 0; i < NS; ++i) mbar_init(&sc_full[i], NDW);
    for (int i = 0; i < NSB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(q_ready, 4);  // the four softmax warps (query rows and zero rows of Q)
    mbar_init(app, NDW);
    mbar_init(drain, 1);
    *s_abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  // The fused call reads tables, row map, frontiers and earlier pages before
  // the programmatic dependency wait (see decode.cuh); q, k, v and every
  // global write come after it.
  const bool early = a.k_new != nullptr;
  if (!early) griddep_wait();
  griddep_launch_dependents();
  if (tid < a.B) {
    const int F = a.frontiers[tid], row = a.table_rows[tid];
    const bool ok = F >= 0 && F <= a.L * 64 && row >= 0 && row < a.C && (a.k_new == nullptr || F >= a.T);
    if (!ok && blockIdx.x == 0 && h == 0) set_status(a.status, NK_STATUS_FRONTIER);
    s_F[tid] = ok ? F : 0;
    s_row[tid] = ok ? row : 0;
  }
  if (warp == 0) {
    tc::alloc(tslot, 512);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;

  // ---- the split plan of decode.cuh --------------------------------------------
  int total = 0, maxp = 0;
  for (int bb = 0; bb < a.B; ++bb) {
    const int np = (s_F[bb] + 63) >> 6;
    total += np;
    maxp = max(maxp, np);
  }
  const int chunk = wave_chunk(s_F, a.B, total, maxp, a.target);
  int b = -1, split = 0, nsplit = 0, npages = 0;
  {
    int acc = 0;
    for (int bb = 0; bb < a.B; ++bb) {
      const int np = (s_F[bb] + 63) >> 6;
      const int ns = max(1, (np + chunk - 1) / chunk);
      if (static_cast<int>(blockIdx.x) < acc + ns) {
        b = bb;
        split = blockIdx.x - acc;
        nsplit = ns;
        npages = np;
        break;
      }
      acc += ns;
    }
  }
  const int F = b >= 0 ? s_F[b] : 0;
  const int p0 = split * chunk;
  const int n = b >= 0 ? min(chunk, npages - p0) : 0;  // pages of this CTA
  const int nt = (n + PPT - 1) / PPT;                  // key tiles
  const int app_lo = early ? (F - a.T) >> 6 : 0x7fffffff;
  const int R_real = a.T * a.G;
  const int32_t* trow = a.tables + static_cast<int64_t>(b >= 0 ? s_row[b] : 0) * a.L;

  if (b < 0) {
    // no work: only the TMEM allocation is released below
  } else if (warp == 12) {
    // -------------------- TMA producer of raw code / scale pages --------------------
    if (lane == 0) {
      bool app_seen = false;
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        int g = trow[p0 + i];
        if (g < 0 || g >= a.M) {
          set_status(a.status, NK_STATUS_PAGE_RANGE);
          g = 0;
        }
        const int s = i % NR;
        if (p0 + i >= app_lo && !app_seen) {  // this page receives new tokens: wait for them
          app_seen = true;
          if (!mbar_wait_bounded(app, 0, a.status)) { *s_abort = 1; break; }
        }
        if (i >= NR && !mbar_wait_bounded(&raw_empty[s], ((i / NR) - 1) & 1, a.status)) { *s_abort = 1; break; }
        uint8_t* st = smem + s * Cfg::RAW;
        const int y = static_cast<int>(tile_row(g, h, a.H, a.M, a.head_major));
        mbar_arrive_expect_tx(&raw_full[s], Cfg::TX);
#pragma unroll
        for (int c = 0; c < Cfg::KCB / Cfg::K_RB; ++c)
          tma_load_2d(st + c * 64 * Cfg::K_RB, &tmk, c * Cfg::K_RB, y, &raw_full[s]);
#pragma unroll
        for (int c = 0; c < Cfg::VCB / Cfg::V_RB; ++c)
          tma_load_2d(st + Cfg::R_KS + c * 64 * Cfg::V_RB, &tmv, c * Cfg::V_RB, y, &raw_full[s]);
        bulk_load(st + Cfg::R_KSC, a.ks + static_cast<int64_t>(y) * Cfg::KSB, 64 * Cfg::KSB, &raw_full[s]);
        bulk_load(st + Cfg::R_VSC, a.vs + static_cast<int64_t>(y) * Cfg::VSB, 64 * Cfg::VSB, &raw_full[s]);
        ++issued;
      }
      // after an abort, the copies still in flight land before the CTA exits
      for (int i = issued > NR ? issued - NR : 0; i < issued; ++i)
        mbar_wait_bounded(&raw_full[i % NR], (i / NR) & 1, a.status, 100000000ull);
    }
  } else if (warp == 13) {
    // ------------------------------ MMA issuer --------------------------------
    // The whole warp runs the loop, so the operand descriptors are warp-uniform
    // values; lane 0 issues every MMA and commit, so a commit covers all MMAs
    // issued before it.
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(q_ready, 0, a.status));
    tc::fence_after();
    const uint32_t k_base = smem_u32(sKf), v_base = smem_u32(sVf);
    // issue order S(0), then S(j), P V(j - 1) for every tile j
    for (int j = 0; ok && j < nt + 1; ++j) {
      if (j < nt) {
        const int ks = j % NK, sb = j % NSB;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&kf_full[ks], (j / NK) & 1, a.status) && !*s_abort);
        if (!ok) break;
        tc::fence_after();
        const uint64_t kd = tc::smem_desc(k_base + ks * Cfg::F16, 16, 1024);
        const uint32_t sd = tmem + Cfg::COL_S + TK * sb;
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc::mma_ts(sd, tmem + Cfg::COL_Q + kk * 8,
                       kd + static_cast<uint64_t>(((kk >> 2) * Cfg::CHUNK + (kk & 3) * 32) >> 4), Cfg::ID_S, kk > 0);
          tc::commit(&s_full[sb]);
          tc::commit(&kf_empty[ks]);
        }
        __syncwarp();
      }
      if (j >= 1) {
        const int jj = j - 1, vs = jj % NV, pb = jj % NSB;
        ok = mbar_wait_bounded(&vf_full[vs], (jj / NV) & 1, a.status) && !*s_abort;
        if (ok) ok = mbar_wait_bounded(&p_full[pb], (jj / NSB) & 1, a.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc::fence_after();
        const uint64_t vd = tc::smem_desc(v_base + vs * Cfg::F16, Cfg::CHUNK, 1024);
        const uint32_t pa = tmem + Cfg::COL_S + TK * pb;
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < TK / 16; ++kk)
            tc::mma_ts(tmem + Cfg::COL_O, pa + kk * 8, vd + static_cast<uint64_t>((kk * 2048) >> 4), Cfg::ID_O,
                       (jj > 0 || kk > 0));
          tc::commit(&o_done[pb]);
          tc::commit(&vf_empty[vs]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      if (!ok) *s_abort = 1;
      tc::commit(drain);
    }
  } else if (warp >= 4) {
    // ----------------- dequantize warps (and the fused append) ------------------
    const int dw = warp - 4;          // 0..7
    const int dt = dw * 32 + lane;    // 0..255
    const int pu = dt % (D / 8), r0 = dt / (D / 8);
    const int k_src = raw_off<KK, D>(r0, pu), v_src = raw_off<KV, D>(r0, pu);
    const int k_dst = f16_off<TK>(r0, pu);
    // V rows are permuted inside 16-row groups: with RPT a multiple of 16 the
    // thread's units still sit at fixed strides from its first one
    const int v_dst = f16_off<TK>(vrow(r0), pu);
    if (early) griddep_wait();
    if (early) {  // the new tokens whose pages this CTA reads, one warp per token
      constexpr int KCBW = code_row_bytes<KK>(D), VCBW = code_row_bytes<KV>(D);
      constexpr int KSBW = scale_row_bytes<KK>(D), VSBW = scale_row_bytes<KV>(D);
      for (int t = dw; t < a.T; t += NDW) {
        const int pos = F - a.T + t, pg = pos >> 6;
        if (pg < p0 || pg >= p0 + n) continue;
        const int g = trow[pg];
        if (g < 0 || g >= a.M) {
          if (lane == 0) set_status(a.status, NK_STATUS_PAGE_RANGE);
          continue;
        }
        const int64_t token_row = tile_row(g, h, a.H, a.M, a.head_major) + (pos & 63);
        const int64_t src = ((static_cast<int64_t>(b) * a.T + t) * a.H + h) * D;
        encode_row<KK, D>(a.k_new + src, a.kc_w + token_row * KCBW, a.ks_w + token_row * KSBW, lane);
        encode_row<KV, D>(a.v_new + src, a.vc_w + token_row * VCBW, a.vs_w + token_row * VSBW, lane);
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncwarp();
      if (lane == 0) v_arrive(app);
    }
    for (int j = 0; j < nt; ++j) {
      const int npg = min(PPT, n - PPT * j);                // pages of this tile
      const int kv_lim = min(F - 64 * (p0 + PPT * j), 64 * npg);  // keys of the tile below the frontier
      bool ok = true;
      const uint8_t* st[PPT];
#pragma unroll
      for (int pi = 0; pi < PPT; ++pi) {
        const int i = PPT * j + min(pi, npg - 1);
        st[pi] = smem + (i % NR) * Cfg::RAW;
        if (pi < npg && ok) ok = mbar_wait_bounded(&raw_full[i % NR], (i / NR) & 1, a.status) && !*s_abort;
      }
      // The tile's key factors and value scales first.  Slot j % NS was last
      // read by the softmax for tile j - NS, which finished before P V(j - NS)
      // could start; tile j - 1 of this loop waited for P V(j - 1 - NV), a
      // later one (commits of one issuing thread complete in order).
      if (ok && dt < TK) {
        float* sc = sSc + (j % NS) * 2 * TK;
        const int pi = dt / 64, row = dt % 64;
        const uint8_t* sp = smem + ((PPT * j + pi) % NR) * Cfg::RAW;  // read only when pi < npg
        float kscale = 1.f, vscale = 1.f;
        if (pi < npg) {
          if constexpr (KK == KIND_FP8)
            kscale = __half2float(*reinterpret_cast<const __half*>(sp + Cfg::R_KSC + row * 2));
          if constexpr (KV == KIND_FP8)
            vscale = __half2float(*reinterpret_cast<const __half*>(sp + Cfg::R_VSC + row * 2));
        }
        sc[dt] = kscale * a.softmax_scale * kLog2e;
        sc[TK + dt] = dt < kv_lim ? vscale : 0.f;
      }
      __syncwarp();
      if (lane == 0) v_arrive(&sc_full[j % NS]);
      // K buffer j % NK held tile j - NK, whose S was issued before
      // P V(j - NK - 1), which tile j - 1 of this loop waited for; only tile
      // NK has no such earlier wait
      static_assert(NS >= NV + 1 && NK == NV, "the waits these orderings rely on");
      if (ok && j == NK) ok = mbar_wait_bounded(&kf_empty[0], 0, a.status);
      if (ok) {
        uint8_t* kt = sKf + (j % NK) * Cfg::F16;
        RawUnit ru[PPT * Cfg::PASSES];
#pragma unroll
        for (int pi = 0; pi < PPT; ++pi)
#pragma unroll
          for (int k = 0; k < Cfg::PASSES; ++k)
            if (pi < npg)  // keys of a missing page are masked in the softmax
              ru[pi * Cfg::PASSES + k] =
                  ld_unit<KK>(st[pi] + k_src + Cfg::RPT * k * Cfg::K_RB,
                              st[pi] + Cfg::R_KSC + (r0 + Cfg::RPT * k) * Cfg::KSB + pu / 2);
#pragma unroll
        for (int pi = 0; pi < PPT; ++pi)
#pragma unroll
          for (int k = 0; k < Cfg::PASSES; ++k)
            if (pi < npg) cvt_unit<KK>(ru[pi * Cfg::PASSES + k], kt + k_dst + 64 * pi * 128 + Cfg::RPT * k * 128, false);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      __syncwarp();
      if (lane == 0) v_arrive(&kf_full[j % NK]);
      if (ok && j >= NV) ok = mbar_wait_bounded(&vf_empty[j % NV], ((j / NV) - 1) & 1, a.status);
      if (ok) {
        uint8_t* vt = sVf + (j % NV) * Cfg::F16;
        RawUnit ru[PPT * Cfg::PASSES];
#pragma unroll
        for (int pi = 0; pi < PPT; ++pi)
#pragma unroll
          for (int k = 0; k < Cfg::PASSES; ++k)
            if (64 * pi + r0 + Cfg::RPT * k < kv_lim)
              ru[pi * Cfg::PASSES + k] =
                  ld_unit<KV>(st[pi] + Cfg::R_KS + v_src + Cfg::RPT * k * Cfg::V_RB,
                              st[pi] + Cfg::R_VSC + (r0 + Cfg::RPT * k) * Cfg::VSB + pu / 2);
#pragma unroll
        for (int pi = 0; pi < PPT; ++pi)
#pragma unroll
          for (int k = 0; k < Cfg::PASSES; ++k) {
            const int key = 64 * pi + r0 + Cfg::RPT * k;
            const int off = Cfg::RPT % 16 == 0 ? v_dst + (64 * pi + Cfg::RPT * k) * 128 : f16_off<TK>(vrow(key), pu);
            cvt_unit<KV>(ru[pi * Cfg::PASSES + k], vt + off, key >= kv_lim);
          }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      __syncwarp();
      if (lane == 0) v_arrive(&vf_full[j % NV]);
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int pi = 0; pi < PPT; ++pi)
          if (pi < npg) v_arrive(&raw_empty[(PPT * j + pi) % NR]);
      }
      if (!ok) {
        *s_abort = 1;
        break;
      }
    }
  } else {
    // ---------- softmax and output: warp w owns query rows [8 w, 8 w + 8) ----------
    constexpr int NREP = TK / 8;                // 16x256b repetitions of a tile's S: 8 keys each
    const int s4 = lane & 3, rl = lane >> 2;    // this thread: row rl of the quadrant, keys 8k + 2 s4 + {0, 1}
    const uint32_t lb = static_cast<uint32_t>(warp * 32) << 16;
    const int qr = 8 * warp + rl;
    const bool row_real = qr < R_real;
    const int lim = F - a.T + qr / a.G;  // keys <= lim are visible to this query row
    if (early) griddep_wait();
    float rs_q = 1.f;  // 2^-e of query row 8 w + lane (lanes 0..7)
    {
      const int myq = 8 * warp + lane;
      const bool q_real = lane < 8 && myq < R_real;
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + ((static_cast<int64_t>(b) * a.T + myq / a.G) * a.Hq + h * a.G + myq % a.G) * D);
      float mx = 0.f;
      if (q_real)
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
      rs_q = ldexpf(1.f, -e);
#pragma unroll 1
      for (int c0 = 0; c0 < D / 2; c0 += 32) {  // lanes 8..31 write zero rows
        uint32_t qv[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = q_real ? src[c0 / 4 + u] : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
            qv[4 * u + k] = pack_f16x2(__low2float(v) * qf, __high2float(v) * qf);
          }
        }
        tc::st32(tmem + lb + Cfg::COL_Q + c0, qv);
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) v_arrive(q_ready);
    }
    const float rs = __shfl_sync(0xffffffffu, rs_q, rl);
    float m_used = -INFINITY, l = 0.f;
    int k_run = KV == KIND_FP8 ? kVLiftInit : 0;  // FP8-row V: the weights, l and O carry 2^k_run (v_lift)
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int sb = j % NSB, ss = j % NS;
      ok = mbar_wait_bounded(&s_full[sb], (j / NSB) & 1, a.status) && !*s_abort;
      if (ok) ok = mbar_wait_bounded(&sc_full[ss], (j / NS) & 1, a.status) && !*s_abort;
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        *s_abort = 1;
        break;
      }
      tc::fence_after();
      float x[2 * NREP];
      {
        uint32_t v[NREP / 8][32];
#pragma unroll
        for (int hh = 0; hh < NREP / 8; ++hh) tc::ld16x256_x8(tmem + lb + Cfg::COL_S + TK * sb + 64 * hh, v[hh]);
        tc::wait_ld();
#pragma unroll
        for (int hh = 0; hh < NREP / 8; ++hh)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            x[16 * hh + 2 * k] = __uint_as_float(v[hh][4 * k]);
            x[16 * hh + 2 * k + 1] = __uint_as_float(v[hh][4 * k + 1]);
          }
      }
      const float* ksc = sSc + ss * 2 * TK + 2 * s4;  // + 8 k: factors of keys 8k + 2 s4 + {0, 1}
      const int kt0 = 64 * (p0 + PPT * j);
      const int key_end = 64 * (p0 + min(PPT * j + PPT, n));  // keys of this CTA in the tile end here
      if (kt0 + TK - 1 <= F - a.T && kt0 + TK <= key_end) {  // every key visible to every row
#pragma unroll
        for (int k = 0; k < NREP; ++k) {
          const float2 kf = *reinterpret_cast<const float2*>(ksc + 8 * k);
          x[2 * k] = row_real ? x[2 * k] * kf.x : -INFINITY;
          x[2 * k + 1] = row_real ? x[2 * k + 1] * kf.y : -INFINITY;
        }
      } else {
        const int kmax = row_real ? min(lim, key_end - 1) - (kt0 + 2 * s4) : -1;
#pragma unroll
        for (int k = 0; k < NREP; ++k) {
          const float2 kf = *reinterpret_cast<const float2*>(ksc + 8 * k);
          x[2 * k] = 8 * k <= kmax ? x[2 * k] * kf.x : -INFINITY;
          x[2 * k + 1] = 8 * k + 1 <= kmax ? x[2 * k + 1] * kf.y : -INFINITY;
        }
      }
      // row maximum: a tree over this thread's keys, then over the row's 4 threads
      float mt[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mt[u] = x[u];
#pragma unroll
      for (int u = 8; u < 2 * NREP; ++u) mt[u & 7] = fmaxf(mt[u & 7], x[u]);
      float pm = fmaxf(fmaxf(fmaxf(mt[0], mt[1]), fmaxf(mt[2], mt[3])), fmaxf(fmaxf(mt[4], mt[5]), fmaxf(mt[6], mt[7])));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
      const float rmax = pm == -INFINITY ? -INFINITY : pm * rs;
      // FP8-row V: the lift of the largest value scale so far (the tile's
      // scales are read across the warp, zero past the frontier)
      int knew = k_run;
      if constexpr (KV == KIND_FP8) {
        const float* vs_all = sSc + ss * 2 * TK + TK;
        float smax = 0.f;
#pragma unroll
        for (int i = 0; i < TK / 32; ++i) smax = fmaxf(smax, vs_all[32 * i + lane]);
        knew = v_lift(__reduce_max_sync(0xffffffffu, __float_as_uint(smax)), k_run);
      }
      // p = 2^(z - m + K): a rescale when the maximum passes the lazy
      // threshold or the lift drops
      float factor = 1.f;
      const float mnew = fmaxf(m_used, rmax);
      bool resc = false;
      if (mnew != -INFINITY && (m_used == -INFINITY || mnew > m_used + Cfg::THR || knew != k_run)) {
        factor = m_used == -INFINITY ? 0.f : ex2((m_used - mnew) + static_cast<float>(knew - k_run));
        m_used = mnew;
        resc = true;
      }
      k_run = knew;
      const float mu = m_used == -INFINITY ? 0.f : m_used - static_cast<float>(k_run);
      uint32_t pk[NREP * 2];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < NREP; ++k) {
        float p0v = ex2(fmaf(x[2 * k], rs, -mu));
        float p1v = ex2(fmaf(x[2 * k + 1], rs, -mu));
        ps[k & 3] += p0v + p1v;
        if constexpr (KV == KIND_FP8) {
          const float2 vf = *reinterpret_cast<const float2*>(ksc + TK + 8 * k);
          p0v *= vf.x;
          p1v *= vf.y;
        }
        // S repetition k -> P columns 8 (k / 2) + 2 s4 + (k % 2) of lane rl
        pk[4 * (k >> 1) + (k & 1)] = pack_f16x2(p0v, p1v);
      }
#pragma unroll
      for (int jj = 0; jj < NREP / 2; ++jj) {  // lanes 8..15 of the quadrant: zero rows
        pk[4 * jj + 2] = 0u;
        pk[4 * jj + 3] = 0u;
      }
      l = l * factor + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      // O is rescaled only when a row's maximum moved: then P V(j - 1) must
      // have landed first (P V(j - 1 - NSB) has, as S(j) has completed, so
      // the parity of o_done[(j - 1) % NSB] is unambiguous); P V(j) waits
      // for this warp's P either way
      if (__any_sync(0xffffffffu, resc && j >= 1)) {
        const int jp = j - 1;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&o_done[jp % NSB], (jp / NSB) & 1, a.status) && !*s_abort);
        if (!ok) {
          *s_abort = 1;
          break;
        }
        tc::fence_after();
        const float f = (resc && j >= 1) ? factor : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t ov[32];
          tc::ld16x256_x8(tmem + lb + Cfg::COL_O + c0, ov);
          tc::wait_ld();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            ov[4 * k] = __float_as_uint(__uint_as_float(ov[4 * k]) * f);
            ov[4 * k + 1] = __float_as_uint(__uint_as_float(ov[4 * k + 1]) * f);
          }
          tc::st16x256_x8(tmem + lb + Cfg::COL_O + c0, ov);
        }
      }
      if constexpr (TK == 128) {
        tc::st16x256_x8(tmem + lb + Cfg::COL_S + TK * sb, pk);
      } else {
        tc::st16x256_x4(tmem + lb + Cfg::COL_S + TK * sb, pk);
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) v_arrive(&p_full[sb]);
    }
    // every MMA of the CTA has completed once drain has (committed after the last P V)
    if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(drain, 0, a.status) && !*s_abort);
    tc::fence_after();
    // row sums over the row's 4 threads (fixed order), then lane L < 8 writes row 8 w + L
    float lr = l + __shfl_xor_sync(0xffffffffu, l, 1);
    lr += __shfl_xor_sync(0xffffffffu, lr, 2);
    const float lt = __shfl_sync(0xffffffffu, lr, 4 * (lane & 7));
    const float m_eff = m_used == -INFINITY ? -INFINITY : m_used - static_cast<float>(k_run);
    const float mt_row = __shfl_sync(0xffffffffu, m_eff, 4 * (lane & 7));
    const int orow = 8 * warp + lane;
    const bool out_real = lane < 8 && orow < R_real;
    const int ot = orow / a.G, og = orow % a.G;
    if (ok) {
      // the split's result: final out / lse (one split) or the partial (m, l, acc)
      const bool final_out = nsplit == 1;
      const int64_t part = (static_cast<int64_t>(b) * a.H + h) * a.target + split;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        if (n > 0) {
          tc::ld32(tmem + lb + Cfg::COL_O + c0, ov);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = 0u;
        }
        if (!out_real) continue;
        if (final_out) {
          __nv_bfloat16* dst = a.out + ((static_cast<int64_t>(b) * a.T + ot) * a.Hq + h * a.G + og) * D + c0;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(dst + 8 * c) = make_uint4(
                pack_bf16x2(__uint_as_float(ov[8 * c]) * inv, __uint_as_float(ov[8 * c + 1]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * c + 2]) * inv, __uint_as_float(ov[8 * c + 3]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * c + 4]) * inv, __uint_as_float(ov[8 * c + 5]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * c + 6]) * inv, __uint_as_float(ov[8 * c + 7]) * inv));
        } else {
          float* dst = a.ws_acc + (part * R + orow) * D + c0;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(dst + 4 * c) = make_uint4(ov[4 * c], ov[4 * c + 1], ov[4 * c + 2], ov[4 * c + 3]);
        }
      }
      if (out_real) {
        if (final_out) {
          if (a.lse)
            a.lse[(static_cast<int64_t>(b) * a.T + ot) * a.Hq + h * a.G + og] =
                lt > 0.f ? (mt_row + log2f(lt)) * kLn2 : -INFINITY;
        } else {
          a.ws_ml[part * R + orow] = make_float2(n > 0 ? mt_row : -INFINITY, n > 0 ? lt : 0.f);
        }
      }
    }
  }

  if (warp == 0 && lane == 0 && b >= 0) mbar_wait_bounded(drain, 0, a.status, 200000000ull);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// Transposed form for head_dim 64 and 128:  S^T = K Q^T,  O^T = V^T P^T.
//
// A tile's 128 keys are the M = 128 rows of both MMAs and its 32 query rows
// are N = 32, so no part of either product is spent on padding rows.  The
// dequantizing warps write the tile's f16 keys straight into tensor memory,
// where they are the A operand of S^T; Q (one power-of-two scale for all the
// CTA's rows) is the K-major B operand in shared memory.  V^T is the A
// operand read MN-major from the f16 V tile, P^T the K-major B operand that
// the softmax warps write to shared memory.  TMEM: K tiles from column 0
// (D / 2 columns each), then the S^T buffers (32 columns each) and O^T
// (lane = dimension, column = query row).
//
// Each softmax warp owns the 32 keys of its lane quadrant, for all 32 query
// rows (thread = key, register n = row n).  Row maxima cross the four warps
// through shared memory once per tile (lane n of each warp reduces row n over
// its keys; a bounded mbarrier collects the four); every warp then holds the
// same running maximum of every row and rescales its own quadrant of O^T when
// it moves.  Row sums stay per thread until the end.
template <int KK, int KV, int D>
struct VTCfg {
  static constexpr int THREADS = 448, NDW = 8;
  static constexpr int TK = 128, PPT = 2;
  static constexpr int RPT = 2048 / D, PASSES = 64 / RPT;  // V units, as in VCfg
  static constexpr int KCB = code_row_bytes<KK>(D), VCB = code_row_bytes<KV>(D);
  static constexpr int KSB = scale_row_bytes<KK>(D), VSB = scale_row_bytes<KV>(D);
  static constexpr int K_RB = KCB < 128 ? KCB : 128, V_RB = VCB < 128 ? VCB : 128;
  static constexpr int R_KS = align_up(64 * KCB, 1024);
  static constexpr int R_KSC = R_KS + align_up(64 * VCB, 1024);
  static constexpr int R_VSC = R_KSC + align_up(64 * KSB, 128);
  static constexpr int RAW = align_up(R_VSC + 64 * VSB, 1024);
  static constexpr int TX = 64 * (KCB + VCB + KSB + VSB);
  static constexpr int F16V = TK * D * 2, CHUNK = TK * 128;  // V tile: D / 64 chunks of TK rows x 128 B
  static constexpr int QB = 32 * D * 2, QCHUNK = 32 * 128;   // Q: D / 64 chunks of 32 rows x 128 B
  static constexpr int PB = 32 * TK * 2, PCHUNK = 32 * 128;  // P^T: TK / 64 chunks of 32 rows x 128 B
  static constexpr int NK = 2, NV = 2, NS = 4, NSB = 2;
  static constexpr int FIXED = NV * F16V + 2 * QB + NSB * PB + NS * 2 * TK * 4 + 4 * 128 * 4 + 2048;
  static constexpr int NR_FIT = (204 * 1024 - FIXED) / RAW;
  static constexpr int NR = NR_FIT > 8 ? 8 : NR_FIT;
  // V tiles first: at D = 64 the M = 128 A operand of O^T also reads the
  // 16 KB after a tile (dimensions 64..127, whose O^T lanes are never read),
  // which the raw stages provide
  static constexpr int OFF_VF = 0;
  static constexpr int OFF_RAW = NV * F16V;
  static constexpr int OFF_Q = OFF_RAW + NR * RAW;
  static constexpr int OFF_P = OFF_Q + 2 * QB;             // Q: two buffers (this piece, the next)
  static constexpr int OFF_SC = OFF_P + NSB * PB;         // [NS][2 TK] float: key factors, value scales
  static constexpr int OFF_MX = OFF_SC + NS * 2 * TK * 4;  // [2][4][32] float: row maxima of each warp
  static constexpr int OFF_L = OFF_MX + 2 * 128 * 4;      // [4][32] float: row sums of each warp
  static constexpr int OFF_MN = OFF_L + 128 * 4;          // [4][32] float: each warp's -(row maxima)
  static constexpr int OFF_FL = OFF_MN + 128 * 4;         // [2][4] int: each warp's "a maximum moved" flag
  static constexpr int OFF_BAR = OFF_FL + 128;
  static constexpr int NBAR = 2 * NR + 2 * NK + 2 * NV + NS + 3 * NSB + 11;
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 128 + 1024;
  static constexpr int SMEM = SMEM_USED > 116 * 1024 ? SMEM_USED : 116 * 1024;
  static constexpr uint32_t COL_K = 0, COL_S = NK * D / 2, COL_O = COL_S + NSB * 32;
  static constexpr uint32_t ID_S = tc::idesc_f16(128, 32, false, false);
  static constexpr uint32_t ID_O = tc::idesc_f16(128, 32, true, false);
  static constexpr float THR = 8.f;  // lazy rescale threshold (log2 units): p <= 2^8
  static_assert(D == 64 || D == 128, "transposed form");
  static_assert(NR >= 2 * PPT && NR * RAW >= CHUNK, "raw stages");
  static_assert(COL_O + 32 <= 512, "TMEM columns");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
  static_assert(RPT * (D / 8) == 32 * NDW && PASSES * RPT == 64 && RPT % 8 == 0, "unit map");
};

// Lane l returns the maximum (MAX) or the sum of a[l] over the warp's lanes,
// a[n] being this lane's value of row n: five exchange stages, each halving
// the rows a lane keeps.
template <bool MAX>
__device__ __forceinline__ float xreduce32(const float (&a)[32], int lane) {
  float r[16];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float send = up ? a[i] : a[i + 16];
      const float keep = up ? a[i + 16] : a[i];
      const float o = __shfl_xor_sync(0xffffffffu, send, 16);
      r[i] = MAX ? fmaxf(keep, o) : keep + o;
    }
  }
#pragma unroll
  for (int s = 8; s >= 1; s >>= 1) {
    const bool up = lane & s;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = up ? r[i] : r[i + s];
      const float keep = up ? r[i + s] : r[i];
      const float o = __shfl_xor_sync(0xffffffffu, send, s);
      r[i] = MAX ? fmaxf(keep, o) : keep + o;
    }
  }
  return r[0];
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Converts this thread's D / 2 key codes (dims [D/2 hd, D/2 hd + D/2) of page
// row `row`) into D / 4 words of f16 pairs.
template <int KIND, int D, int RB>
__device__ __forceinline__ void key_half_f16(const uint8_t* stage, const uint8_t* scales, int row, int hd,
                                             uint32_t (&w)[D / 4]) {
  if constexpr (KIND == KIND_FP8) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {  // 16 codes per load
      const int col = (D / 2) * hd + 16 * c;
      const uint4 x = *reinterpret_cast<const uint4*>(stage + (col / RB) * (64 * RB) + swz<RB>(row, col % RB));
      e4m3x4_f16(x.x, w[8 * c + 0], w[8 * c + 1]);
      e4m3x4_f16(x.y, w[8 * c + 2], w[8 * c + 3]);
      e4m3x4_f16(x.z, w[8 * c + 4], w[8 * c + 5]);
      e4m3x4_f16(x.w, w[8 * c + 6], w[8 * c + 7]);
    }
  } else {
    uint32_t sc4;  // the E4M3 scales of the half's D / 32 groups of 16
    if constexpr (D == 128) {
      sc4 = *reinterpret_cast<const uint32_t*>(scales + 4 * hd);
    } else {
      sc4 = *reinterpret_cast<const uint16_t*>(scales + 2 * hd);
    }
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {  // 32 codes (two groups) per load
      const int col = (D / 4) * hd + 16 * c;
      const uint4 x = *reinterpret_cast<const uint4*>(stage + (col / RB) * (64 * RB) + swz<RB>(row, col % RB));
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint32_t sb = (sc4 >> (8 * (2 * c + g))) & 0xFFu;
        const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint16_t>(sb * 0x101u));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t* o = &w[16 * c + 8 * g + 4 * h];
          e2m1x8_f16(xs[2 * g + h], o[0], o[1], o[2], o[3]);
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = hmul2_u32(o[i], s2);
        }
      }
    }
  }
}

// One piece of a head's work: pages [p0, p0 + n) of row b, piece k of ns.
// A head's rows are cut in row order into pieces of `chunk` pages
// (piece_chunk: about total / a.nseg, or one wave-filling split per CTA when
// that would make pieces short); CTA x of gridDim.x takes pieces
// [x S / gridDim.x, (x + 1) S / gridDim.x) of the S pieces.
struct VSeg {
  int b, k, ns, p0, n, F;
};

__device__ __forceinline__ VSeg vt_seg(int sg, const int* s_F, int B, int chunk) {
  VSeg r{0, 0, 1, 0, 0, 0};
  int acc = 0;
  for (int bb = 0; bb < B; ++bb) {
    const int np = (s_F[bb] + 63) >> 6;
    const int ns = max(1, (np + chunk - 1) / chunk);
    if (sg < acc + ns) {
      r.b = bb;
      r.k = sg - acc;
      r.ns = ns;
      r.p0 = r.k * chunk;
      r.n = min(chunk, np - r.p0);
      r.F = s_F[bb];
      return r;
    }
    acc += ns;
  }
  return r;
}

template <int KK, int KV, int D>
__global__ void __launch_bounds__(448, 1)
    vtdecode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, DecodeArgs a) {
  using Cfg = VTCfg<KK, KV, D>;
  constexpr int NR = Cfg::NR, NK = Cfg::NK, NV = Cfg::NV, NS = Cfg::NS, NDW = Cfg::NDW, NSB = Cfg::NSB;
  constexpr int TK = Cfg::TK, PPT = Cfg::PPT;
  constexpr int R = 32;  // query rows of a part in the workspace
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sVf = smem + Cfg::OFF_VF;
  uint8_t* sRaw = smem + Cfg::OFF_RAW;
  uint8_t* sQ = smem + Cfg::OFF_Q;  // [2][QB]: the Q of pieces i and i + 1
  uint8_t* sP = smem + Cfg::OFF_P;
  float* sSc = reinterpret_cast<float*>(smem + Cfg::OFF_SC);
  float* sMx = reinterpret_cast<float*>(smem + Cfg::OFF_MX);
  float* sL = reinterpret_cast<float*>(smem + Cfg::OFF_L);
  float* sMn = reinterpret_cast<float*>(smem + Cfg::OFF_MN);
  int* sFl = reinterpret_cast<int*>(smem + Cfg::OFF_FL);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* raw_full = bars;             // [NR] raw page stages
  uint64_t* raw_empty = raw_full + NR;
  uint64_t* kf_full = raw_empty + NR;    // [NK] f16 K tiles (TMEM)
  uint64_t* kf_empty = kf_full + NK;
  uint64_t* vf_full = kf_empty + NK;     // [NV] f16 V tiles
  uint64_t* vf_empty = vf_full + NV;
  uint64_t* sc_full = vf_empty + NV;     // [NS] key factors / value scales of a tile
  uint64_t* s_full = sc_full + NS;       // [NSB]: S^T(J) in buffer J % NSB
  uint64_t* p_full = s_full + NSB;       // [NSB]: P^T(J) in shared buffer J % NSB
  uint64_t* o_done = p_full + NSB;       // [NSB]: O^T += V^T P^T(J) done
  uint64_t* mx_full = o_done + NSB;      // [2]: the four warps' row maxima, exchange e in slot e % 2
  uint64_t* fl_full = mx_full + 2;       // [2]: the four warps' flags, exchange e in slot e % 2
  uint64_t* q_ready = fl_full + 2;       // [2]: Q of piece i in buffer i % 2
  uint64_t* seg_done = q_ready + 2;      // every MMA of a piece completed (one phase per piece)
  uint64_t* o_free = seg_done + 1;       // the softmax warps have read a piece's O^T
  uint64_t* app = o_free + 1;
  uint64_t* drain = app + 1;
  uint64_t* fin = drain + 1;             // the four warps' row sums (one phase per piece)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
  int* s_F = reinterpret_cast<int*>(tslot + 2);     // [8]
  int* s_row = s_F + 8;                             // [8]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  if (tid == 0) {
    for (int i = 0; i < NR; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], NDW);
    }
    for (int i = 0; i < NK; ++i) {
      mbar_init(&kf_full[i], NDW);
      mbar_init(&kf_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&vf_full[i], NDW);
      mbar_init(&vf_empty[i], 1);
    }
    for (int i = 0; i < NS; ++i) mbar_init(&sc_full[i], NDW);
    for (int i = 0; i < NSB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&o_done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&mx_full[i], 4);
      mbar_init(&fl_full[i], 4);
      mbar_init(&q_ready[i], 4);
    }
    mbar_init(seg_done, 1);
    mbar_init(o_free, 4);
    mbar_init(app, NDW);
    mbar_init(drain, 1);
    mbar_init(fin, 4);
    *s_abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  const bool early = a.k_new != nullptr;
  if (!early) griddep_wait();
  griddep_launch_dependents();
  if (tid < a.B) {
    const int F = a.frontiers[tid], row = a.table_rows[tid];
    const bool ok = F >= 0 && F <= a.L * 64 && row >= 0 && row < a.C && (a.k_new == nullptr || F >= a.T);
    if (!ok && blockIdx.x == 0 && h == 0) set_status(a.status, NK_STATUS_FRONTIER);
    s_F[tid] = ok ? F : 0;
    s_row[tid] = ok ? row : 0;
  }
  if (warp == 0) {
    tc::alloc(tslot, 512);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;

  // ---- the pieces of this CTA --------------------------------------------------
  int total = 0, maxp = 0;
  for (int bb = 0; bb < a.B; ++bb) {
    const int np = (s_F[bb] + 63) >> 6;
    total += np;
    maxp = max(maxp, np);
  }
  const int chunk = piece_chunk(s_F, a, total, maxp);
  int nsegs = 0;
  for (int bb = 0; bb < a.B; ++bb) nsegs += max(1, (((s_F[bb] + 63) >> 6) + chunk - 1) / chunk);
  const int s_lo = static_cast<int>(static_cast<int64_t>(blockIdx.x) * nsegs / gridDim.x);
  const int s_hi = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * nsegs / gridDim.x);
  const int R_real = a.T * a.G;
  auto trow_of = [&](int bb) { return a.tables + static_cast<int64_t>(s_row[bb]) * a.L; };

  if (s_hi <= s_lo) {
    // no work: only the TMEM allocation is released below
  } else if (warp == 12) {
    // -------------------- TMA producer of raw code / scale pages --------------------
    if (lane == 0) {
      bool app_seen = false, ok = true;
      int issued = 0;  // pages of the CTA so far: the stage ring runs across pieces
      for (int sg = s_lo; ok && sg < s_hi; ++sg) {
        const VSeg g0 = vt_seg(sg, s_F, a.B, chunk);
        const int32_t* trow = trow_of(g0.b);
        const int app_lo = early ? (g0.F - a.T) >> 6 : 0x7fffffff;
        for (int i = 0; i < g0.n; ++i) {
          int g = trow[g0.p0 + i];
          if (g < 0 || g >= a.M) {
            set_status(a.status, NK_STATUS_PAGE_RANGE);
            g = 0;
          }
          const int s = issued % NR;
          if (g0.p0 + i >= app_lo && !app_seen) {  // this page receives new tokens: wait for them
            app_seen = true;
            if (!mbar_wait_bounded(app, 0, a.status)) { *s_abort = 1; ok = false; break; }
          }
          if (issued >= NR && !mbar_wait_bounded(&raw_empty[s], ((issued / NR) - 1) & 1, a.status)) {
            *s_abort = 1;
            ok = false;
            break;
          }
          uint8_t* st = sRaw + s * Cfg::RAW;
          const int y = static_cast<int>(tile_row(g, h, a.H, a.M, a.head_major));
          mbar_arrive_expect_tx(&raw_full[s], Cfg::TX);
#pragma unroll
          for (int c = 0; c < Cfg::KCB / Cfg::K_RB; ++c)
            tma_load_2d(st + c * 64 * Cfg::K_RB, &tmk, c * Cfg::K_RB, y, &raw_full[s]);
#pragma unroll
          for (int c = 0; c < Cfg::VCB / Cfg::V_RB; ++c)
            tma_load_2d(st + Cfg::R_KS + c * 64 * Cfg::V_RB, &tmv, c * Cfg::V_RB, y, &raw_full[s]);
          bulk_load(st + Cfg::R_KSC, a.ks + static_cast<int64_t>(y) * Cfg::KSB, 64 * Cfg::KSB, &raw_full[s]);
          bulk_load(st + Cfg::R_VSC, a.vs + static_cast<int64_t>(y) * Cfg::VSB, 64 * Cfg::VSB, &raw_full[s]);
          ++issued;
        }
      }
      // after an abort, the copies still in flight land before the CTA exits
      for (int i = issued > NR ? issued - NR : 0; i < issued; ++i)
        mbar_wait_bounded(&raw_full[i % NR], (i / NR) & 1, a.status, 100000000ull);
    }
  } else if (warp == 13) {
    // ------------------------------ MMA issuer --------------------------------
    // converged warp, lane 0 issues every MMA and commit (see vdecode_kernel).
    // Tiles are numbered J across the CTA's pieces; within a piece the issue
    // order is S^T(0), then S^T(j), O^T += V^T P^T(j - 1) for every tile j.
    bool ok = true;
    const uint32_t v_base = smem_u32(sVf), p_base = smem_u32(sP);
    int J = 0;
    for (int sg = s_lo; ok && sg < s_hi; ++sg) {
      const int i = sg - s_lo;  // piece of this CTA
      const int nt = (vt_seg(sg, s_F, a.B, chunk).n + PPT - 1) / PPT;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&q_ready[i & 1], (i >> 1) & 1, a.status) && !*s_abort);
      if (!ok) break;
      tc::fence_after();
      const uint64_t qd = tc::smem_desc(smem_u32(sQ) + (i & 1) * Cfg::QB, 16, 1024);
      // O^T of the previous piece must have been read before this piece's
      // first O^T += V^T P^T overwrites it
      bool o_waited = i == 0;
      for (int j = 0; ok && j < nt + 1; ++j) {
        if (j < nt) {
          const int jg = J + j, ks = jg % NK, sb = jg % NSB;
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&kf_full[ks], (jg / NK) & 1, a.status) && !*s_abort);
          if (!ok) break;
          tc::fence_after();
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc::mma_ts(tmem + Cfg::COL_S + 32 * sb, tmem + Cfg::COL_K + ks * (D / 2) + kk * 8,
                         qd + static_cast<uint64_t>(((kk >> 2) * Cfg::QCHUNK + (kk & 3) * 32) >> 4), Cfg::ID_S,
                         kk > 0);
            tc::commit(&s_full[sb]);
            tc::commit(&kf_empty[ks]);
          }
          __syncwarp();
        }
        if (j >= 1) {
          const int jj = j - 1, jg = J + jj, vs = jg % NV, pb = jg % NSB;
          if (!o_waited) {
            o_waited = true;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_free, (i - 1) & 1, a.status) && !*s_abort);
            if (!ok) break;
          }
          ok = mbar_wait_bounded(&vf_full[vs], (jg / NV) & 1, a.status) && !*s_abort;
          if (ok) ok = mbar_wait_bounded(&p_full[pb], (jg / NSB) & 1, a.status);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc::fence_after();
          const uint64_t vd = tc::smem_desc(v_base + vs * Cfg::F16V, Cfg::CHUNK, 1024);
          const uint64_t pd = tc::smem_desc(p_base + pb * Cfg::PB, 16, 1024);
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < TK / 16; ++kk)
              tc::mma_ss(tmem + Cfg::COL_O, vd + static_cast<uint64_t>((kk * 2048) >> 4),
                         pd + static_cast<uint64_t>(((kk >> 2) * Cfg::PCHUNK + (kk & 3) * 32) >> 4), Cfg::ID_O,
                         (jj > 0 || kk > 0));
            tc::commit(&o_done[pb]);
            tc::commit(&vf_empty[vs]);
          }
          __syncwarp();
        }
      }
      if (ok && !o_waited)  // a piece without pages still keeps the o_free phases in step
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_free, (i - 1) & 1, a.status) && !*s_abort);
      if (lane == 0) tc::commit(seg_done);
      __syncwarp();
      J += nt;
    }
    if (lane == 0) {
      if (!ok) *s_abort = 1;
      tc::commit(drain);
    }
  } else if (warp >= 4) {
    // ----------------- dequantize warps (and the fused append) ------------------
    const int dw = warp - 4;          // 0..7
    const int dt = dw * 32 + lane;    // 0..255
    const int pu = dt % (D / 8), r0 = dt / (D / 8);
    const int v_src = raw_off<KV, D>(r0, pu);
    const int v_dst = f16_off<TK>(r0, pu);
    // K: this warp writes the TMEM lanes of its quadrant (keys 32 (warp % 4) +
    // lane of the tile), dims [D/2 hd, D/2 hd + D/2)
    const int kq = warp & 3, hd = dw >> 2;
    const int kpg = kq >> 1, krow = 32 * (kq & 1) + lane;  // page of the tile, row in the page
    const uint32_t k_taddr = tmem + (static_cast<uint32_t>(32 * kq) << 16) + Cfg::COL_K + (D / 4) * hd;
    if (early) griddep_wait();
    if (early) {  // the new tokens whose pages this CTA reads, one warp per token
      constexpr int KCBW = code_row_bytes<KK>(D), VCBW = code_row_bytes<KV>(D);
      constexpr int KSBW = scale_row_bytes<KK>(D), VSBW = scale_row_bytes<KV>(D);
      for (int sg = s_lo; sg < s_hi; ++sg) {
        const VSeg g0 = vt_seg(sg, s_F, a.B, chunk);
        const int32_t* trow = trow_of(g0.b);
        for (int t = dw; t < a.T; t += NDW) {
          const int pos = g0.F - a.T + t, pg = pos >> 6;
          if (pg < g0.p0 || pg >= g0.p0 + g0.n) continue;
          const int g = trow[pg];
          if (g < 0 || g >= a.M) {
            if (lane == 0) set_status(a.status, NK_STATUS_PAGE_RANGE);
            continue;
          }
          const int64_t token_row = tile_row(g, h, a.H, a.M, a.head_major) + (pos & 63);
          const int64_t src = ((static_cast<int64_t>(g0.b) * a.T + t) * a.H + h) * D;
          encode_row<KK, D>(a.k_new + src, a.kc_w + token_row * KCBW, a.ks_w + token_row * KSBW, lane);
          encode_row<KV, D>(a.v_new + src, a.vc_w + token_row * VCBW, a.vs_w + token_row * VSBW, lane);
        }
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncwarp();
      if (lane == 0) v_arrive(app);
    }
    bool ok = true;
    int J = 0, ip = 0;  // tiles and pages of the CTA before this piece
    for (int sg = s_lo; ok && sg < s_hi; ++sg) {
      const VSeg g0 = vt_seg(sg, s_F, a.B, chunk);
      const int n = g0.n, nt = (n + PPT - 1) / PPT;
      for (int j = 0; j < nt; ++j) {
        const int jg = J + j;
        const int npg = min(PPT, n - PPT * j);                          // pages of this tile
        const int kv_lim = min(g0.F - 64 * (g0.p0 + PPT * j), 64 * npg);  // keys of the tile below the frontier
        const uint8_t* st[PPT];
#pragma unroll
        for (int pi = 0; pi < PPT; ++pi) {
          const int ig = ip + PPT * j + min(pi, npg - 1);
          st[pi] = sRaw + (ig % NR) * Cfg::RAW;
          if (pi < npg && ok) ok = mbar_wait_bounded(&raw_full[ig % NR], (ig / NR) & 1, a.status) && !*s_abort;
        }
        // the tile's key factors and value scales (slot reuse as in vdecode_kernel)
        if (ok && dt < TK) {
          float* sc = sSc + (jg % NS) * 2 * TK;
          const int pi = dt / 64, row = dt % 64;
          const uint8_t* sp = sRaw + ((ip + PPT * j + pi) % NR) * Cfg::RAW;  // read only when pi < npg
          float kscale = 1.f, vscale = 1.f;
          if (pi < npg) {
            if constexpr (KK == KIND_FP8)
              kscale = __half2float(*reinterpret_cast<const __half*>(sp + Cfg::R_KSC + row * 2));
            if constexpr (KV == KIND_FP8)
              vscale = __half2float(*reinterpret_cast<const __half*>(sp + Cfg::R_VSC + row * 2));
          }
          sc[dt] = kscale * a.softmax_scale * kLog2e;
          sc[TK + dt] = dt < kv_lim ? vscale : 0.f;
        }
        __syncwarp();
        if (lane == 0) v_arrive(&sc_full[jg % NS]);
        // K buffer J % NK is free once S^T(J - NK) has completed.  (The scale
        // slot J % NS is free as in vdecode_kernel: P V runs in order of J,
        // across pieces too.)
        static_assert(NS >= NV + 1, "the scale-slot ordering");
        if (ok && jg >= NK) ok = mbar_wait_bounded(&kf_empty[jg % NK], ((jg / NK) - 1) & 1, a.status);
        ok = __all_sync(0xffffffffu, ok);
        if (ok && kpg < npg) {  // keys of a missing page are masked in the softmax
          uint32_t kw[D / 4];
          const uint8_t* ks = kpg == 0 ? st[0] : st[1];  // no run-time index into st
          key_half_f16<KK, D, Cfg::K_RB>(ks, ks + Cfg::R_KSC + krow * Cfg::KSB, krow, hd, kw);
          if constexpr (D == 128) {
            tc::st32(k_taddr + (jg % NK) * (D / 2), kw);
          } else {
            tc::st16(k_taddr + (jg % NK) * (D / 2), kw);
          }
          tc::wait_st();
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) v_arrive(&kf_full[jg % NK]);
        if (ok && jg >= NV) ok = mbar_wait_bounded(&vf_empty[jg % NV], ((jg / NV) - 1) & 1, a.status);
        if (ok) {
          uint8_t* vt = sVf + (jg % NV) * Cfg::F16V;
          RawUnit ru[PPT * Cfg::PASSES];
#pragma unroll
          for (int pi = 0; pi < PPT; ++pi)
#pragma unroll
            for (int k = 0; k < Cfg::PASSES; ++k)
              if (64 * pi + r0 + Cfg::RPT * k < kv_lim)
                ru[pi * Cfg::PASSES + k] =
                    ld_unit<KV>(st[pi] + Cfg::R_KS + v_src + Cfg::RPT * k * Cfg::V_RB,
                                st[pi] + Cfg::R_VSC + (r0 + Cfg::RPT * k) * Cfg::VSB + pu / 2);
#pragma unroll
          for (int pi = 0; pi < PPT; ++pi)
#pragma unroll
            for (int k = 0; k < Cfg::PASSES; ++k) {
              const int key = 64 * pi + r0 + Cfg::RPT * k;
              cvt_unit<KV>(ru[pi * Cfg::PASSES + k], vt + v_dst + (64 * pi + Cfg::RPT * k) * 128, key >= kv_lim);
            }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) v_arrive(&vf_full[jg % NV]);
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int pi = 0; pi < PPT; ++pi)
            if (pi < npg) v_arrive(&raw_empty[(ip + PPT * j + pi) % NR]);
        }
        if (!ok) {
          *s_abort = 1;
          break;
        }
      }
      J += nt;
      ip += n;
    }
  } else {
    // ---- softmax and output: warp w owns keys [32 w, 32 w + 32) of every tile ----
    const int kq = 32 * warp + lane;  // this thread's key in a tile
    const uint32_t lq = static_cast<uint32_t>(32 * warp) << 16;
    if (early) griddep_wait();
    // Q of piece sg into buffer qb: one power-of-two scale 2^e for its query
    // rows (returned: 2^-e); this warp writes rows [8 w, 8 w + 8) of the
    // K-major B operand
    auto write_q = [&](int sg, int qb) -> float {
      const int bq = vt_seg(sg, s_F, a.B, chunk).b;
      auto qrow = [&](int r) {
        return a.q + ((static_cast<int64_t>(bq) * a.T + r / a.G) * a.Hq + h * a.G + r % a.G) * D;
      };
      float mx = 0.f;
      for (int u = lane; u < R_real * (D / 8); u += 32) {
        const uint4 x = *reinterpret_cast<const uint4*>(qrow(u / (D / 8)) + 8 * (u % (D / 8)));
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&x);
#pragma unroll
        for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fabsf(__bfloat162float(e[k])));
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      int ex = 0;
      if (mx > 0.f) frexpf(mx, &ex);
      const int e = mx > 0.f ? min(15 - ex, 100) : 0;  // 2^e stays finite in fp32
      const float qf = ldexpf(1.f, e);
      uint8_t* qbuf = sQ + qb * Cfg::QB;
      for (int u = lane; u < 8 * (D / 8); u += 32) {
        const int r = 8 * warp + u / (D / 8), c = u % (D / 8);
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (r < R_real) x = *reinterpret_cast<const uint4*>(qrow(r) + 8 * c);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
          o[k] = pack_f16x2(__low2float(v) * qf, __high2float(v) * qf);
        }
        *reinterpret_cast<uint4*>(qbuf + (c / 8) * Cfg::QCHUNK + swz<128>(r, (c % 8) * 16)) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) v_arrive(&q_ready[qb]);
      return ldexpf(1.f, -e);
    };
    float rs_cur = write_q(s_lo, 0);
    float rs_next = s_lo + 1 < s_hi ? write_q(s_lo + 1, 1) : 1.f;
    // P^T (K-major, 32 query rows x TK keys): element (row r, key kq)
    const uint32_t p_col = smem_u32(sP) + (kq / 64) * Cfg::PCHUNK;
    const int p_byte = (kq % 64) * 2;
    // -(running maximum of row r), 0 while it is -inf: this warp's copy, written by lane r
    float* mn = sMn + 32 * warp;
    int nfull = 0, nflag = 0;  // exchanges of row maxima and of flags so far
    bool ok = true;
    int J = 0;
    for (int sg = s_lo; ok && sg < s_hi; ++sg) {
      const int i = sg - s_lo;
      const VSeg g0 = vt_seg(sg, s_F, a.B, chunk);
      const int n = g0.n, nt = (n + PPT - 1) / PPT, F = g0.F, p0 = g0.p0;
      const float rs = rs_cur;
      mn[lane] = 0.f;
      __syncwarp();
      float lacc[32];  // row sums of this thread's key
#pragma unroll
      for (int r = 0; r < 32; ++r) lacc[r] = 0.f;
      float m_self = -INFINITY;        // the running maximum of row `lane`
      uint32_t inf_rows = 0xffffffffu;  // rows whose running maximum is still -inf
      int k_run = KV == KIND_FP8 ? kVLiftInit : 0;  // FP8-row V: the weights and O^T carry 2^k_run (v_lift)
      for (int j = 0; j < nt; ++j) {
        const int jg = J + j, sb = jg % NSB, ss = jg % NS;
        ok = mbar_wait_bounded(&s_full[sb], (jg / NSB) & 1, a.status) && !*s_abort;
        if (ok) ok = mbar_wait_bounded(&sc_full[ss], (jg / NS) & 1, a.status) && !*s_abort;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          *s_abort = 1;
          break;
        }
        tc::fence_after();
        // t[r] = z - m of row r for this key: z = s * key factor * 2^-e, m the
        // running maximum (0 while -inf); -inf where the key is masked
        float t[32];
        {
          uint32_t v[32];
          tc::ld32(tmem + lq + Cfg::COL_S + 32 * sb, v);
          tc::wait_ld();
          const float kfr = sSc[ss * 2 * TK + kq] * rs;
          const int kt0 = 64 * (p0 + PPT * j);
          const int key_end = 64 * (p0 + min(PPT * j + PPT, n));  // keys of this piece in the tile end here
          const bool all_vis = kt0 + TK - 1 <= F - a.T && kt0 + TK <= key_end;  // every key visible to every row
          const int key = kt0 + kq, d = key - (F - a.T);
          // key k is visible to rows r with r / G >= k - (F - T)
          const int rmin = all_vis ? 0 : (key >= key_end ? 32 : (d <= 0 ? 0 : min(32, a.G * d)));
#pragma unroll
          for (int r4 = 0; r4 < 32; r4 += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mn + r4);
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              t[r4 + q4] = r4 + q4 >= rmin ? fmaf(__uint_as_float(v[r4 + q4]), kfr, mm[q4]) : -INFINITY;
          }
        }
        // Does a row's maximum move past the lazy threshold (or leave -inf)?
        // A piece's first tile always sets the maxima; later tiles exchange
        // one flag per warp and take the exact per-row reduction only when one
        // is set.
        bool full = j == 0;
        if (!full) {
          float tm = t[0];
#pragma unroll
          for (int r = 1; r < 32; ++r) tm = fmaxf(tm, t[r]);
          bool fl = tm > Cfg::THR;
          if (inf_rows != 0u) {
#pragma unroll
            for (int r = 0; r < 32; ++r) fl |= ((inf_rows >> r) & 1u) && t[r] > -INFINITY;
          }
          fl = __any_sync(0xffffffffu, fl);
          const int e = nflag++;
          int* fls = sFl + (e & 1) * 4;
          if (lane == 0) {
            fls[warp] = fl ? 1 : 0;
            v_arrive(&fl_full[e & 1]);
          }
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(&fl_full[e & 1], (e >> 1) & 1, a.status) && !*s_abort)) {
            ok = false;
            *s_abort = 1;
            break;
          }
          const int4 f4 = *reinterpret_cast<const int4*>(fls);
          full = (f4.x | f4.y | f4.z | f4.w) != 0;
        }
        bool moved = false;
        float fac = 1.f;
        if (full) {
          // exact row maxima: this warp's over lanes, then the four warps' through shared memory
          float* mx = sMx + (nfull & 1) * 128;
          mx[32 * warp + lane] = xreduce32<true>(t, lane);
          __syncwarp();
          if (lane == 0) v_arrive(&mx_full[nfull & 1]);
          if (!__all_sync(0xffffffffu,
                          mbar_wait_bounded(&mx_full[nfull & 1], (nfull >> 1) & 1, a.status) && !*s_abort)) {
            ok = false;
            *s_abort = 1;
            break;
          }
          const float gm = fmaxf(fmaxf(mx[lane], mx[32 + lane]), fmaxf(mx[64 + lane], mx[96 + lane]));
          ++nfull;
          const float mcur = m_self == -INFINITY ? 0.f : m_self;  // the value t is relative to
          const float mnew = fmaxf(m_self, gm + mcur);
          const bool resc = mnew != -INFINITY && (m_self == -INFINITY || mnew > m_self + Cfg::THR);
          if (resc) {
            fac = m_self == -INFINITY ? 0.f : ex2(m_self - mnew);
            m_self = mnew;
          }
          const float mneg_new = m_self == -INFINITY ? 0.f : -m_self;
          const float delta = mneg_new + mcur;  // t of row `lane` moves by this
          mn[lane] = mneg_new;
          inf_rows = __ballot_sync(0xffffffffu, m_self == -INFINITY);
          moved = __any_sync(0xffffffffu, resc);
          if (moved) {
#pragma unroll
            for (int r = 0; r < 32; ++r) {
              lacc[r] *= __shfl_sync(0xffffffffu, fac, r);
              t[r] += __shfl_sync(0xffffffffu, delta, r);
            }
          }
          __syncwarp();
        }
        // P = 2^t, stored as f16 into column kq of the K-major P^T tile
        const uint32_t pb = p_col + sb * Cfg::PB;
        float vsc = 1.f;
        int knew = k_run;
        if constexpr (KV == KIND_FP8) {
          // the lift of the largest value scale so far (the tile's scales
          // are read across the warp, zero past the frontier); l stays unlifted
          const float* vs_all = sSc + ss * 2 * TK + TK;
          float smax = 0.f;
#pragma unroll
          for (int u = 0; u < TK / 32; ++u) smax = fmaxf(smax, vs_all[32 * u + lane]);
          knew = v_lift(__reduce_max_sync(0xffffffffu, __float_as_uint(smax)), k_run);
          vsc = vs_all[kq] * pow2i(knew);
        }
#pragma unroll
        for (int r = 0; r < 32; r += 2) {
          const float p0v = ex2(t[r]), p1v = ex2(t[r + 1]);
          lacc[r] += p0v;
          lacc[r + 1] += p1v;
          const uint32_t w = KV == KIND_FP8 ? pack_f16x2(p0v * vsc, p1v * vsc) : pack_f16x2(p0v, p1v);
          st_shared_u16(pb + swz<128>(r, p_byte), static_cast<uint16_t>(w & 0xFFFFu));
          st_shared_u16(pb + swz<128>(r + 1, p_byte), static_cast<uint16_t>(w >> 16));
        }
        if ((moved || knew != k_run) && j >= 1) {
          // O^T is rescaled only when a row's maximum moved or the lift
          // dropped: O^T += V^T P^T(J - 1) must have landed first (the one
          // before it has, as S^T(J) has completed); O^T += V^T P^T(J) waits
          // for this warp's P^T
          const float kf = pow2i(knew - k_run);
          const int jp = jg - 1;
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(&o_done[jp % NSB], (jp / NSB) & 1, a.status) && !*s_abort)) {
            ok = false;
            *s_abort = 1;
            break;
          }
          tc::fence_after();
#pragma unroll
          for (int c0 = 0; c0 < 32; c0 += 16) {
            uint32_t ov[16];
            tc::ld16(tmem + lq + Cfg::COL_O + c0, ov);
            tc::wait_ld();
#pragma unroll
            for (int r = 0; r < 16; ++r)
              ov[r] = __float_as_uint(__uint_as_float(ov[r]) * (__shfl_sync(0xffffffffu, fac, c0 + r) * kf));
            tc::st16(tmem + lq + Cfg::COL_O + c0, ov);
          }
          tc::wait_st();
        }
        k_run = knew;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc::fence_before();
        __syncwarp();
        if (lane == 0) v_arrive(&p_full[sb]);
      }
      if (!ok) break;
      // the piece's result: every MMA of it has completed once seg_done has
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(seg_done, i & 1, a.status) && !*s_abort);
      tc::fence_after();
      sL[32 * warp + lane] = xreduce32<false>(lacc, lane);
      __syncwarp();
      if (lane == 0) v_arrive(fin);
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(fin, i & 1, a.status) && !*s_abort);
      if (!ok) break;
      {
        const float lt = (sL[lane] + sL[32 + lane]) + (sL[64 + lane] + sL[96 + lane]);  // row `lane`
        const int b = g0.b;
        const bool final_out = g0.ns == 1;
        const int64_t part = (static_cast<int64_t>(b) * a.H + h) * a.target + g0.k;
        const float unlift = KV == KIND_FP8 ? pow2i(-k_run) : 1.f;  // O^T carries 2^k_run
        const float inv_self = lt > 0.f ? unlift / lt : 0.f;
        const int dim = 32 * warp + lane;  // O^T lane: the dimension this thread writes
        uint32_t ov[32];
        if (n > 0) {
          tc::ld32(tmem + lq + Cfg::COL_O, ov);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int r = 0; r < 32; ++r) ov[r] = 0u;
        }
        // O^T and sL are read: the next piece may overwrite both
        tc::fence_before();
        __syncwarp();
        if (lane == 0) v_arrive(o_free);
        if (32 * warp < D) {  // at D = 64 the lanes of quadrants 2 and 3 hold no dimension
#pragma unroll
          for (int r = 0; r < 32; ++r) {
            const float inv = __shfl_sync(0xffffffffu, inv_self, r);
            if (r < R_real) {
              const int ot = r / a.G, og = r % a.G;
              if (final_out) {
                a.out[((static_cast<int64_t>(b) * a.T + ot) * a.Hq + h * a.G + og) * D + dim] =
                    __float2bfloat16_rn(__uint_as_float(ov[r]) * inv);
              } else {
                a.ws_acc[(part * R + r) * D + dim] = __uint_as_float(ov[r]) * unlift;
              }
            }
          }
        }
        if (warp == 0 && lane < R_real) {
          const int ot = lane / a.G, og = lane % a.G;
          if (final_out) {
            if (a.lse)
              a.lse[(static_cast<int64_t>(b) * a.T + ot) * a.Hq + h * a.G + og] =
                  lt > 0.f ? (m_self + log2f(lt)) * kLn2 : -INFINITY;
          } else {
            a.ws_ml[part * R + lane] = make_float2(n > 0 ? m_self : -INFINITY, n > 0 ? lt : 0.f);
          }
        }
      }
      J += nt;
      // Q buffer i % 2 is free (every S^T of this piece has completed): the
      // Q of piece i + 2 goes there
      rs_cur = rs_next;
      if (sg + 2 < s_hi) rs_next = write_q(sg + 2, i & 1);
    }
  }

  if (warp == 0 && lane == 0 && s_hi > s_lo) mbar_wait_bounded(drain, 0, a.status, 200000000ull);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::dealloc(tmem, 512);
}

template <int KK, int KV, int D>
static cudaError_t launch_v(const nk_pool* p, int layer, const DecodeArgs& a, dim3 grid, cudaStream_t s) {
  using Cfg = VCfg<KK, KV, D>;
  auto k = vdecode_kernel<KK, KV, D>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaError_t e = launch_pdl(k, grid, dim3(Cfg::THREADS), Cfg::SMEM, s, p->tmap[layer * 2 + 0], p->tmap[layer * 2 + 1], a);
  if (e != cudaSuccess) return e;
  return launch_pdl(merge_kernel<D, 4>, dim3(a.B, a.H, D / 32), dim3(256), 0, s, a);
}

template <int KK, int KV, int D>
static cudaError_t launch_vt(const nk_pool* p, int layer, const DecodeArgs& a, dim3 grid, cudaStream_t s) {
  using Cfg = VTCfg<KK, KV, D>;
  auto k = vtdecode_kernel<KK, KV, D>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaError_t e = launch_pdl(k, grid, dim3(Cfg::THREADS), Cfg::SMEM, s, p->tmap[layer * 2 + 0], p->tmap[layer * 2 + 1], a);
  if (e != cudaSuccess) return e;
  return launch_pdl(merge_kernel<D, 4>, dim3(a.B, a.H, D / 32), dim3(256), 0, s, a);
}

template <int KK, int KV>
static cudaError_t vdispatch(const nk_pool* p, int layer, const DecodeArgs& a, int nqt, dim3 grid, cudaStream_t s) {
  if (nqt != 4) return cudaErrorInvalidValue;
  switch (p->desc.head_dim) {
    case 64: return launch_vt<KK, KV, 64>(p, layer, a, grid, s);
    case 128: return launch_vt<KK, KV, 128>(p, layer, a, grid, s);
    case 256: return launch_v<KK, KV, 256>(p, layer, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

DecodeFn vdecode_for(int profile, int D, int nqt) {
  if (nqt != 4 || (D != 64 && D != 128 && D != 256)) return nullptr;
  switch (profile) {
    case NK_FP8_E4M3_ROW: return vdispatch<KIND_FP8, KIND_FP8>;
    case NK_NVFP4_G16: return vdispatch<KIND_NVFP4, KIND_NVFP4>;
    case NK_K8V4: return vdispatch<KIND_FP8, KIND_NVFP4>;
    default: return nullptr;
  }
}

}  // namespace nk
