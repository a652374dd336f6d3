// decode.cuh -- split-K paged GQA decode / verify attention over the typed
// KV pool (kernel template; instantiated per profile in decode_*.cu).
//
// Contract ("Paged KV cache" maintainer design page, consumer view section):
// the consumer reads K/V pages in place through block_tables[table_rows[b]],
// translating logical block -> physical page once per page (never in the
// inner loop), with no gather-to-contiguous copy; a frontier may sit at any
// offset of the last page and bytes past it are never used.
//
// Work split.  A CTA (4 warps) owns one (row b, KV head h, page range).  The
// page ranges come from the device-side frontiers, so the host needs no
// lengths and the launch is graph-stable: with N_b = ceil(F_b / 64) pages,
// every CTA computes chunk = ceil(sum_b N_b / target), row b gets
// ceil(N_b / chunk) splits, and CTA x of a head takes the x-th split.
//
// Per page (64 keys), staged by TMA into a ring of NSTAGE shared buffers:
//  QK:  warp w takes keys [16w, 16w+16): S^T(16 keys x R queries) via
//       mma.m16n8k16 with the K tile as the A operand (ldmatrix of the raw
//       codes, exact conversion to f16/bf16 in registers) and q as B.
//       INT8-G64 group scales and FP8 row scales multiply the fp32 partial
//       sums; NVFP4 scales multiply the f16 operand (exact product).
//  softmax: base-2 online softmax, CTA-wide running max per query through
//       shared memory; P (f16 / bf16) goes to shared memory.
//  PV:  warp w takes head dims [w*D/4, (w+1)*D/4): O^T += V^T P^T, V^T built
//       in registers from the V tile (ldmatrix.trans for bf16; byte gathers
//       for 8-bit and 4-bit codes), V scales folded in as f16 products.
// The CTA writes unnormalised partials (m, l, acc) to the workspace, or the
// final out / lse when its row has a single split.
#pragma once

#include "device.cuh"
#include "internal.h"

namespace nk {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeArgs {
  const __nv_bfloat16* q;
  const int32_t* tables;
  const int32_t* table_rows;
  const int32_t* frontiers;
  const uint8_t* ks;  // K scale plane of the layer (nullptr for BF16)
  const uint8_t* vs;  // V scale plane
  __nv_bfloat16* out;
  float* lse;
  float2* ws_ml;  // [B][H][maxsplit][R]
  float* ws_acc;  // [B][H][maxsplit][R][D]
  int* status;
  float softmax_scale;
  int B, T, Hq, H, G, L, M, C;
  int target;    // splits per head the chunking aims at (= maxsplit)
};

// Valid length of compact row b.  A table row outside [0, C) or a frontier
// outside [0, L*64] never leads to an out-of-bounds access: the row is read as
// empty and NK_STATUS_FRONTIER is recorded (by one thread, when `flag`).
__device__ __forceinline__ int row_frontier(const DecodeArgs& a, int b, bool flag) {
  const int F = a.frontiers[b];
  const int row = a.table_rows[b];
  if (F < 0 || F > a.L * 64 || row < 0 || row >= a.C) {
    if (flag) set_status(a.status, NK_STATUS_FRONTIER);
    return 0;
  }
  return F;
}

__device__ __forceinline__ int plan_chunk(const DecodeArgs& a, bool flag = false) {
  int total = 0;
  for (int b = 0; b < a.B; ++b) total += (row_frontier(a, b, flag) + 63) >> 6;
  const int chunk = (total + a.target - 1) / a.target;
  return chunk < 1 ? 1 : chunk;
}

template <int KIND>
struct CodeRow {
  static constexpr int bytes(int D) { return KIND == KIND_BF16 ? 2 * D : KIND == KIND_NVFP4 ? D / 2 : D; }
};
template <int KIND>
struct ScaleRow {
  static constexpr int bytes(int D) {
    return KIND == KIND_BF16 ? 0 : KIND == KIND_INT8 ? 2 * (D / 64) : KIND == KIND_FP8 ? 2 : D / 16;
  }
};

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int KK, int KV, int D, int NQT>
struct DecodeCfg {
  static constexpr int R = 8 * NQT;  // query rows (T * G) padded to n-tiles of 8
  static constexpr int KCB = CodeRow<KK>::bytes(D);
  static constexpr int VCB = CodeRow<KV>::bytes(D);
  static constexpr int KSB = ScaleRow<KK>::bytes(D);
  static constexpr int VSB = ScaleRow<KV>::bytes(D);
  static constexpr int K_RB = KCB < 128 ? KCB : 128;
  static constexpr int V_RB = VCB < 128 ? VCB : 128;
  static constexpr int K_TILE = 64 * KCB, V_TILE = 64 * VCB;
  static constexpr int KS_TILE = 64 * KSB, VS_TILE = 64 * VSB;
  static constexpr int OFF_V = align_up(K_TILE, 1024);
  static constexpr int OFF_KS = OFF_V + align_up(V_TILE, 1024);
  static constexpr int OFF_VS = OFF_KS + align_up(KS_TILE, 128);
  static constexpr int STAGE = align_up(OFF_VS + VS_TILE, 1024);
  static constexpr int TX_BYTES = K_TILE + V_TILE + KS_TILE + VS_TILE;
  // Ring depth: three 64 KB stages (one CTA per SM) for BF16 D=256, else as
  // many stages as fit in ~104 KB so that two CTAs share an SM.
  static constexpr int NSTAGE =
      STAGE > 48 * 1024 ? 3 : (104 * 1024 / STAGE < 2 ? 2 : (104 * 1024 / STAGE > 8 ? 8 : 104 * 1024 / STAGE));
  static constexpr int P_PITCH = 64 * 2 + 16;  // bytes per query row of P (padded)
  // BF16 pools run PV in bf16: P is kept as hi + lo bf16 parts (about 16
  // significant bits), the f16 paths keep one f16 P.
  static constexpr int NPBUF = (KK == KIND_BF16) ? 2 : 1;
  static constexpr int P_BUF = align_up(R * P_PITCH, 128);
  static constexpr int OFF_P = NSTAGE * STAGE;
  static constexpr int OFF_RED = OFF_P + NPBUF * P_BUF;
  static constexpr int OFF_BAR = OFF_RED + 2 * 4 * R * 4;
  static constexpr int SMEM = OFF_BAR + NSTAGE * 8 + 32 + 1024;  // + alignment slack
  static constexpr bool MMA_BF16 = (KK == KIND_BF16);
  static constexpr int KSTEPS = D / 16;
  static constexpr int DW = D / 4;     // head dims per warp in PV
  static constexpr int MT = DW / 16;   // m-tiles per warp in PV
  static constexpr int EPT = DW >= 32 ? 4 : 2;  // V elements gathered per key per thread
};

// d index of the q element in slot i (0..3: b0.lo, b0.hi, b1.lo, b1.hi) of
// k-step s for lane column c; must match how the K operand is built.
template <int KK>
__device__ __forceinline__ int q_dim(int s, int i, int c) {
  if constexpr (KK == KIND_BF16) return 16 * s + 2 * c + (i & 1) + (i >> 1) * 8;
  else if constexpr (KK == KIND_NVFP4) return 32 * (s >> 1) + 8 * c + 4 * (s & 1) + i;
  else return 16 * s + 4 * c + i;
}

// Converts two codes (bytes 0,1 of w when HI = false, bytes 2,3 when true)
// to an exact f16x2.
template <int KIND, bool HI>
__device__ __forceinline__ uint32_t cvt_pair(uint32_t w) {
  if constexpr (KIND == KIND_INT8) return s8pair_to_f16x2(__byte_perm(w, 0, HI ? 0x3322 : 0x1100));
  else return e4m3x2_to_f16x2(static_cast<uint16_t>(HI ? (w >> 16) : (w & 0xFFFFu)));
}

template <int KK, int KV, int D, int NQT>
__global__ void __launch_bounds__(128)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  DecodeArgs a) {
  using Cfg = DecodeCfg<KK, KV, D, NQT>;
  constexpr int R = Cfg::R;
  constexpr int NSTAGE = Cfg::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Ps = smem + Cfg::OFF_P;
  float* red_max = reinterpret_cast<float*>(smem + Cfg::OFF_RED);  // [4][R]
  float* red_l = red_max + 4 * R;                                  // [4][R]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  int* s_flags = reinterpret_cast<int*>(bars + NSTAGE);             // [0] abort

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int h = blockIdx.y;

  // ---- which (row, split) this CTA owns --------------------------------
  const int chunk = plan_chunk(a, tid == 0 && blockIdx.x == 0 && h == 0);
  int b = -1, split = 0, nsplit = 0, npages = 0;
  {
    int acc = 0;
    for (int bb = 0; bb < a.B; ++bb) {
      const int np = (row_frontier(a, bb, false) + 63) >> 6;
      const int ns = (np + chunk - 1) / chunk;
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
  if (b < 0) return;
  const int F = row_frontier(a, b, false);
  const int p0 = split * chunk;
  const int n = min(chunk, npages - p0);  // pages of this CTA (>= 1)
  const int32_t* table = a.tables + static_cast<int64_t>(a.table_rows[b]) * a.L;
  const int R_real = a.T * a.G;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
    s_flags[0] = 0;
    fence_barrier_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  __syncthreads();

  // Producer: thread 0 stages page p0 + i into stage i % NSTAGE.
  auto issue = [&](int i) {
    const int s = i % NSTAGE;
    int g = table[p0 + i];
    if (g < 0 || g >= a.M) {  // never copy from outside the pool
      set_status(a.status, NK_STATUS_PAGE_RANGE);
      g = 0;                  // the row's result is then undefined
    }
    uint8_t* st = smem + s * Cfg::STAGE;
    const int y = (g * a.H + h) * 64;
    mbar_arrive_expect_tx(&bars[s], Cfg::TX_BYTES);
#pragma unroll
    for (int j = 0; j < Cfg::KCB / Cfg::K_RB; ++j) tma_load_2d(st + j * 64 * Cfg::K_RB, &tmk, j * Cfg::K_RB, y, &bars[s]);
#pragma unroll
    for (int j = 0; j < Cfg::VCB / Cfg::V_RB; ++j)
      tma_load_2d(st + Cfg::OFF_V + j * 64 * Cfg::V_RB, &tmv, j * Cfg::V_RB, y, &bars[s]);
    if constexpr (Cfg::KS_TILE > 0) {
      bulk_load(st + Cfg::OFF_KS, a.ks + static_cast<int64_t>(y) * Cfg::KSB, Cfg::KS_TILE, &bars[s]);
      bulk_load(st + Cfg::OFF_VS, a.vs + static_cast<int64_t>(y) * Cfg::VSB, Cfg::VS_TILE, &bars[s]);
    }
  };
  int issued = 0;
  if (tid == 0) {
    for (; issued < NSTAGE && issued < n; ++issued) issue(issued);
  }

  // ---- q fragments (B operand of QK) ----------------------------------------
  // Quantized profiles run the MMAs in f16: q is scaled by 2^e so that
  // max|q| * 2^e lies in [2^14, 2^15) (exact for every element above
  // max|q| * 2^-31), and the scores divide 2^e back out.
  uint32_t qf[Cfg::KSTEPS][NQT][2];
  float qscale_log2 = 0.f;
  {
    auto qrow_ptr = [&](int j, bool& live) {
      const int qr = 8 * j + r;
      live = qr < R_real;
      const int t = live ? qr / a.G : 0, g = live ? qr % a.G : 0;
      return a.q + ((static_cast<int64_t>(b) * a.T + t) * a.Hq + h * a.G + g) * D;
    };
    float f = 1.f;
    if constexpr (!Cfg::MMA_BF16) {
      float mx = 0.f;
#pragma unroll
      for (int j = 0; j < NQT; ++j) {
        bool live;
        const __nv_bfloat16* qp = qrow_ptr(j, live);
        if (live)
#pragma unroll
          for (int s = 0; s < Cfg::KSTEPS; ++s)
#pragma unroll
            for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fabsf(__bfloat162float(qp[q_dim<KK>(s, i, c)])));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      int ex = 0;
      if (mx > 0.f) frexpf(mx, &ex);
      const int e = mx > 0.f ? 15 - ex : 0;
      f = ldexpf(1.f, e);
      qscale_log2 = static_cast<float>(e);
    }
#pragma unroll
    for (int j = 0; j < NQT; ++j) {
      bool live;
      const __nv_bfloat16* qp = qrow_ptr(j, live);
#pragma unroll
      for (int s = 0; s < Cfg::KSTEPS; ++s) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = live ? __bfloat162float(qp[q_dim<KK>(s, i, c)]) * f : 0.f;
        if constexpr (Cfg::MMA_BF16) {
          qf[s][j][0] = pack_bf16x2(v[0], v[1]);
          qf[s][j][1] = pack_bf16x2(v[2], v[3]);
        } else {
          qf[s][j][0] = pack_f16x2(v[0], v[1]);
          qf[s][j][1] = pack_f16x2(v[2], v[3]);
        }
      }
    }
  }
  const float sc = a.softmax_scale * kLog2e * exp2f(-qscale_log2);

  // ---- running state -----------------------------------------------------
  float m_run[NQT][2], l_part[NQT][2];
  float o[Cfg::MT][NQT][4];
#pragma unroll
  for (int j = 0; j < NQT; ++j) {
    m_run[j][0] = m_run[j][1] = -INFINITY;
    l_part[j][0] = l_part[j][1] = 0.f;
  }
#pragma unroll
  for (int mt = 0; mt < Cfg::MT; ++mt)
#pragma unroll
    for (int j = 0; j < NQT; ++j) o[mt][j][0] = o[mt][j][1] = o[mt][j][2] = o[mt][j][3] = 0.f;

  // query-token limits: query row q may see keys <= F - T + q / G (and < F)
  int lim[NQT][2];
#pragma unroll
  for (int j = 0; j < NQT; ++j)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int qr = 8 * j + 2 * c + u;
      lim[j][u] = min(F - a.T + qr / a.G, F - 1);
    }

  bool aborted = false;
  for (int i = 0; i < n; ++i) {
    const int s = i % NSTAGE;
    const uint8_t* st = smem + s * Cfg::STAGE;
    const uint32_t kbase = smem_u32(st);
    const uint32_t vbase = smem_u32(st + Cfg::OFF_V);
    if (!mbar_wait_bounded(&bars[s], (i / NSTAGE) & 1, a.status)) s_flags[0] = 1;
    const int page = p0 + i;
    const int key0 = page * 64;

    // ---------------- QK: S^T for keys [16*warp, 16*warp+16) -------------
    float S[NQT][4];
#pragma unroll
    for (int j = 0; j < NQT; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
    const int krow_ld = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row of this lane
    const int kr0 = 16 * warp + r, kr1 = kr0 + 8;                      // keys of this thread's S rows
    if constexpr (KK == KIND_BF16) {
#pragma unroll
      for (int s16 = 0; s16 < Cfg::KSTEPS; ++s16) {
        const int col = (2 * s16 + (lane >> 4)) * 16;
        const uint32_t addr = kbase + (col / 128) * (64 * 128) + swz<128>(krow_ld, col % 128);
        uint32_t A[4];
        ldsm_x4(addr, A[0], A[1], A[2], A[3]);
#pragma unroll
        for (int j = 0; j < NQT; ++j) mma16816<true>(S[j], A, qf[s16][j][0], qf[s16][j][1]);
      }
    } else if constexpr (KK == KIND_NVFP4) {
      constexpr int RB = Cfg::K_RB;
      const uint8_t* ks_tile = st + Cfg::OFF_KS;
#pragma unroll
      for (int cp = 0; cp < Cfg::KCB / 32; ++cp) {  // chunk pairs (64 dims)
        const int col = (2 * cp + (lane >> 4)) * 16;
        const uint32_t addr = kbase + (col / RB) * (64 * RB) + swz<RB>(krow_ld, col % RB);
        uint32_t d[4];
        ldsm_x4(addr, d[0], d[1], d[2], d[3]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {  // chunk 2cp+u: regs d[2u] (key r), d[2u+1] (key r+8)
          const int cc = 2 * cp + u;
          const int blk = 2 * cc + (c >> 1);
          const __half s0 = __ushort_as_half(static_cast<uint16_t>(
              e4m3x2_to_f16x2(ks_tile[kr0 * Cfg::KSB + blk]) & 0xFFFFu));
          const __half s1 = __ushort_as_half(static_cast<uint16_t>(
              e4m3x2_to_f16x2(ks_tile[kr1 * Cfg::KSB + blk]) & 0xFFFFu));
          const uint32_t sc0 = pack_h2(s0, s0), sc1 = pack_h2(s1, s1);
          const uint32_t w0 = d[2 * u], w1 = d[2 * u + 1];
          uint32_t f0[4], f1[4];
          f0[0] = hmul2_u32(e2m1x2_byte_to_f16x2<0>(w0), sc0);
          f0[1] = hmul2_u32(e2m1x2_byte_to_f16x2<1>(w0), sc0);
          f0[2] = hmul2_u32(e2m1x2_byte_to_f16x2<2>(w0), sc0);
          f0[3] = hmul2_u32(e2m1x2_byte_to_f16x2<3>(w0), sc0);
          f1[0] = hmul2_u32(e2m1x2_byte_to_f16x2<0>(w1), sc1);
          f1[1] = hmul2_u32(e2m1x2_byte_to_f16x2<1>(w1), sc1);
          f1[2] = hmul2_u32(e2m1x2_byte_to_f16x2<2>(w1), sc1);
          f1[3] = hmul2_u32(e2m1x2_byte_to_f16x2<3>(w1), sc1);
          const uint32_t A0[4] = {f0[0], f1[0], f0[1], f1[1]};
          const uint32_t A1[4] = {f0[2], f1[2], f0[3], f1[3]};
#pragma unroll
          for (int j = 0; j < NQT; ++j) {
            mma16816<false>(S[j], A0, qf[2 * cc][j][0], qf[2 * cc][j][1]);
            mma16816<false>(S[j], A1, qf[2 * cc + 1][j][0], qf[2 * cc + 1][j][1]);
          }
        }
      }
    } else {  // INT8 / FP8: 16 dims per 16-byte chunk
      constexpr int RB = Cfg::K_RB;
      constexpr int NCH = Cfg::KCB / 16;
      const uint8_t* ks_tile = st + Cfg::OFF_KS;
      float Sg[NQT][4];
#pragma unroll
      for (int cp = 0; cp < NCH / 2; ++cp) {
        if constexpr (KK == KIND_INT8) {
          if ((cp & 1) == 0) {
#pragma unroll
            for (int j = 0; j < NQT; ++j) Sg[j][0] = Sg[j][1] = Sg[j][2] = Sg[j][3] = 0.f;
          }
        }
        const int col = (2 * cp + (lane >> 4)) * 16;
        const uint32_t addr = kbase + (col / RB) * (64 * RB) + swz<RB>(krow_ld, col % RB);
        uint32_t d[4];
        ldsm_x4(addr, d[0], d[1], d[2], d[3]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int cc = 2 * cp + u;
          const uint32_t A[4] = {cvt_pair<KK, false>(d[2 * u]), cvt_pair<KK, false>(d[2 * u + 1]),
                                 cvt_pair<KK, true>(d[2 * u]), cvt_pair<KK, true>(d[2 * u + 1])};
#pragma unroll
          for (int j = 0; j < NQT; ++j) {
            if constexpr (KK == KIND_INT8) mma16816<false>(Sg[j], A, qf[cc][j][0], qf[cc][j][1]);
            else mma16816<false>(S[j], A, qf[cc][j][0], qf[cc][j][1]);
          }
        }
        if constexpr (KK == KIND_INT8) {
          if ((cp & 1) == 1) {  // end of a 64-dim group: apply its scale
            const int grp = cp >> 1;
            const float g0 = __half2float(*reinterpret_cast<const __half*>(ks_tile + kr0 * Cfg::KSB + 2 * grp));
            const float g1 = __half2float(*reinterpret_cast<const __half*>(ks_tile + kr1 * Cfg::KSB + 2 * grp));
#pragma unroll
            for (int j = 0; j < NQT; ++j) {
              S[j][0] = fmaf(Sg[j][0], g0, S[j][0]);
              S[j][1] = fmaf(Sg[j][1], g0, S[j][1]);
              S[j][2] = fmaf(Sg[j][2], g1, S[j][2]);
              S[j][3] = fmaf(Sg[j][3], g1, S[j][3]);
            }
          }
        }
      }
      if constexpr (KK == KIND_FP8) {
        const float g0 = __half2float(*reinterpret_cast<const __half*>(ks_tile + kr0 * 2));
        const float g1 = __half2float(*reinterpret_cast<const __half*>(ks_tile + kr1 * 2));
#pragma unroll
        for (int j = 0; j < NQT; ++j) {
          S[j][0] *= g0;
          S[j][1] *= g0;
          S[j][2] *= g1;
          S[j][3] *= g1;
        }
      }
    }

    // ---------------- scores, masking, tile max ---------------------------
    const int kg0 = key0 + kr0, kg1 = key0 + kr1;
#pragma unroll
    for (int j = 0; j < NQT; ++j) {
      S[j][0] = kg0 <= lim[j][0] ? S[j][0] * sc : -INFINITY;
      S[j][1] = kg0 <= lim[j][1] ? S[j][1] * sc : -INFINITY;
      S[j][2] = kg1 <= lim[j][0] ? S[j][2] * sc : -INFINITY;
      S[j][3] = kg1 <= lim[j][1] ? S[j][3] * sc : -INFINITY;
      float v0 = fmaxf(S[j][0], S[j][2]), v1 = fmaxf(S[j][1], S[j][3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        v0 = fmaxf(v0, __shfl_xor_sync(0xffffffffu, v0, off));
        v1 = fmaxf(v1, __shfl_xor_sync(0xffffffffu, v1, off));
      }
      if (r == 0) {
        red_max[warp * R + 8 * j + 2 * c] = v0;
        red_max[warp * R + 8 * j + 2 * c + 1] = v1;
      }
    }
    __syncthreads();  // (1) tile maxima visible; stage of page i-1 free
    if (s_flags[0]) {
      aborted = true;
      break;
    }
    if (tid == 0 && i >= 1 && issued < n) issue(issued++);

    // ---------------- online softmax, P to shared memory ---------------------
    float alpha[NQT][2];
#pragma unroll
    for (int j = 0; j < NQT; ++j)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int qr = 8 * j + 2 * c + u;
        float mx = m_run[j][u];
#pragma unroll
        for (int w = 0; w < 4; ++w) mx = fmaxf(mx, red_max[w * R + qr]);
        const float mu = mx == -INFINITY ? 0.f : mx;
        alpha[j][u] = ex2(m_run[j][u] - mu);
        m_run[j][u] = mx;
        const float p_a = ex2(S[j][u] - mu), p_b = ex2(S[j][2 + u] - mu);
        l_part[j][u] = l_part[j][u] * alpha[j][u] + p_a + p_b;
        uint16_t ha, hb;
        if constexpr (Cfg::MMA_BF16) {
          const __nv_bfloat16 a_hi = __float2bfloat16_rn(p_a), b_hi = __float2bfloat16_rn(p_b);
          ha = __bfloat16_as_ushort(a_hi);
          hb = __bfloat16_as_ushort(b_hi);
          const uint16_t la = __bfloat16_as_ushort(__float2bfloat16_rn(p_a - __bfloat162float(a_hi)));
          const uint16_t lb = __bfloat16_as_ushort(__float2bfloat16_rn(p_b - __bfloat162float(b_hi)));
          *reinterpret_cast<uint16_t*>(Ps + Cfg::P_BUF + qr * Cfg::P_PITCH + kr0 * 2) = la;
          *reinterpret_cast<uint16_t*>(Ps + Cfg::P_BUF + qr * Cfg::P_PITCH + kr1 * 2) = lb;
        } else {
          ha = __half_as_ushort(__float2half_rn(p_a));
          hb = __half_as_ushort(__float2half_rn(p_b));
        }
        *reinterpret_cast<uint16_t*>(Ps + qr * Cfg::P_PITCH + kr0 * 2) = ha;
        *reinterpret_cast<uint16_t*>(Ps + qr * Cfg::P_PITCH + kr1 * 2) = hb;
      }
    __syncthreads();  // (2) P complete

    // ---------------- PV: O^T(dims of this warp x R) += V^T P^T ---------------
#pragma unroll
    for (int mt = 0; mt < Cfg::MT; ++mt)
#pragma unroll
      for (int j = 0; j < NQT; ++j) {
        o[mt][j][0] *= alpha[j][0];
        o[mt][j][1] *= alpha[j][1];
        o[mt][j][2] *= alpha[j][0];
        o[mt][j][3] *= alpha[j][1];
      }
    // P^T fragments: pf[buffer][j][ks][0..1] (buffer 1 = low bf16 part)
    uint32_t pf[Cfg::NPBUF][NQT][4][2];
#pragma unroll
    for (int pb = 0; pb < Cfg::NPBUF; ++pb)
#pragma unroll
      for (int j = 0; j < NQT; ++j)
#pragma unroll
        for (int kp = 0; kp < 2; ++kp) {
          const int qrow = 8 * j + (lane & 7);
          const int kcol = 32 * kp + 8 * ((lane >> 3) & 1) + 16 * (lane >> 4);
          ldsm_x4(smem_u32(Ps + pb * Cfg::P_BUF + qrow * Cfg::P_PITCH + kcol * 2), pf[pb][j][2 * kp][0],
                  pf[pb][j][2 * kp][1], pf[pb][j][2 * kp + 1][0], pf[pb][j][2 * kp + 1][1]);
        }
    const int kvalid = F - key0;  // keys >= kvalid of this page are past the frontier
    const int dw0 = warp * Cfg::DW;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      // validity masks of keys (2c, 2c+1) and (2c+8, 2c+9) of this k-step
      uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
      if (kvalid < 64) {
        const int k0 = 16 * ks + 2 * c;
        mlo = (k0 < kvalid ? 0x0000FFFFu : 0u) | (k0 + 1 < kvalid ? 0xFFFF0000u : 0u);
        mhi = (k0 + 8 < kvalid ? 0x0000FFFFu : 0u) | (k0 + 9 < kvalid ? 0xFFFF0000u : 0u);
      }
      if constexpr (KV == KIND_BF16) {
#pragma unroll
        for (int mt = 0; mt < Cfg::MT; ++mt) {
          const int key = 16 * ks + (lane & 7) + ((lane >> 4) & 1) * 8;
          const int col = (dw0 + 16 * mt + 8 * ((lane >> 3) & 1)) * 2;
          const uint32_t addr = vbase + (col / 128) * (64 * 128) + swz<128>(key, col % 128);
          uint32_t A[4];
          ldsm_x4_t(addr, A[0], A[1], A[2], A[3]);
          A[0] &= mlo;
          A[1] &= mlo;
          A[2] &= mhi;
          A[3] &= mhi;
#pragma unroll
          for (int j = 0; j < NQT; ++j) {
            mma16816<true>(o[mt][j], A, pf[0][j][ks][0], pf[0][j][ks][1]);
            mma16816<true>(o[mt][j], A, pf[1][j][ks][0], pf[1][j][ks][1]);
          }
        }
      } else {
        constexpr int RB = Cfg::V_RB;
        constexpr int EPT = Cfg::EPT;
        const int kk0 = 16 * ks + 2 * c;
        const int keys[4] = {kk0, kk0 + 1, kk0 + 8, kk0 + 9};
        const uint8_t* vs_tile = st + Cfg::OFF_VS;
#pragma unroll
        for (int p = 0; p < Cfg::MT / (EPT / 2); ++p) {  // groups of 8*EPT dims
          const int dg = dw0 + 8 * EPT * p;
          const int dthr = dg + EPT * r;  // first dim of this thread in the group
          uint32_t pair_lo[EPT], pair_hi[EPT];
          if constexpr (KV == KIND_NVFP4) {
            // 4-bit codes: EPT dims = EPT/2 bytes per key
            uint32_t f[4][EPT / 2];
#pragma unroll
            for (int kx = 0; kx < 4; ++kx) {
              const int colb = dthr / 2;
              const uint8_t* rowp = reinterpret_cast<const uint8_t*>(st + Cfg::OFF_V) +
                                    (colb / RB) * (64 * RB) + swz<RB>(keys[kx], colb % RB);
              const uint32_t wv = EPT == 4 ? *reinterpret_cast<const uint16_t*>(rowp) : *rowp;
              const __half sv = __ushort_as_half(static_cast<uint16_t>(
                  e4m3x2_to_f16x2(vs_tile[keys[kx] * Cfg::VSB + dthr / 16]) & 0xFFFFu));
              const uint32_t s2 = pack_h2(sv, sv);
              f[kx][0] = hmul2_u32(e2m1x2_byte_to_f16x2<0>(wv), s2);
              if constexpr (EPT == 4) f[kx][1] = hmul2_u32(e2m1x2_byte_to_f16x2<1>(wv), s2);
            }
#pragma unroll
            for (int e2 = 0; e2 < EPT / 2; ++e2) {
              pair_lo[2 * e2] = __byte_perm(f[0][e2], f[1][e2], 0x5410);
              pair_lo[2 * e2 + 1] = __byte_perm(f[0][e2], f[1][e2], 0x7632);
              pair_hi[2 * e2] = __byte_perm(f[2][e2], f[3][e2], 0x5410);
              pair_hi[2 * e2 + 1] = __byte_perm(f[2][e2], f[3][e2], 0x7632);
            }
          } else {
            // 8-bit codes: EPT bytes per key
            uint32_t wv[4];
#pragma unroll
            for (int kx = 0; kx < 4; ++kx) {
              const uint8_t* rowp = reinterpret_cast<const uint8_t*>(st + Cfg::OFF_V) +
                                    (dthr / RB) * (64 * RB) + swz<RB>(keys[kx], dthr % RB);
              wv[kx] = EPT == 4 ? *reinterpret_cast<const uint32_t*>(rowp)
                                : *reinterpret_cast<const uint16_t*>(rowp);
            }
            uint32_t slo, shi;  // (s_key0, s_key1), (s_key8, s_key9) as f16x2
            if constexpr (KV == KIND_INT8) {
              const int grp = dg / 64;
              const uint16_t* sp = reinterpret_cast<const uint16_t*>(vs_tile);
              slo = sp[keys[0] * (Cfg::VSB / 2) + grp] | (uint32_t(sp[keys[1] * (Cfg::VSB / 2) + grp]) << 16);
              shi = sp[keys[2] * (Cfg::VSB / 2) + grp] | (uint32_t(sp[keys[3] * (Cfg::VSB / 2) + grp]) << 16);
            } else {
              const uint16_t* sp = reinterpret_cast<const uint16_t*>(vs_tile);
              slo = sp[keys[0]] | (uint32_t(sp[keys[1]]) << 16);
              shi = sp[keys[2]] | (uint32_t(sp[keys[3]]) << 16);
            }
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
              if constexpr (KV == KIND_INT8) {
                const uint32_t sel = e | (e << 4) | ((4 + e) << 8) | ((4 + e) << 12);
                pair_lo[e] = hmul2_u32(s8pair_to_f16x2(__byte_perm(wv[0], wv[1], sel)), slo);
                pair_hi[e] = hmul2_u32(s8pair_to_f16x2(__byte_perm(wv[2], wv[3], sel)), shi);
              } else {
                const uint32_t sel = e | ((4 + e) << 4);
                pair_lo[e] = hmul2_u32(e4m3x2_to_f16x2(static_cast<uint16_t>(__byte_perm(wv[0], wv[1], sel))), slo);
                pair_hi[e] = hmul2_u32(e4m3x2_to_f16x2(static_cast<uint16_t>(__byte_perm(wv[2], wv[3], sel))), shi);
              }
            }
          }
#pragma unroll
          for (int mg = 0; mg < EPT / 2; ++mg) {
            const uint32_t A[4] = {pair_lo[2 * mg] & mlo, pair_lo[2 * mg + 1] & mlo,
                                   pair_hi[2 * mg] & mhi, pair_hi[2 * mg + 1] & mhi};
            const int mt = p * (EPT / 2) + mg;
#pragma unroll
            for (int j = 0; j < NQT; ++j) mma16816<false>(o[mt][j], A, pf[0][j][ks][0], pf[0][j][ks][1]);
          }
        }
      }
    }
  }

  if (aborted) {
    if (tid == 0) {  // drain the copies still in flight (bounded)
      for (int i = 0; i < issued; ++i) mbar_wait_bounded(&bars[i % NSTAGE], (i / NSTAGE) & 1, a.status, 100000000ull);
    }
    return;
  }

  // ---- final reductions of l over the 8 lanes of a column and the 4 warps ---
#pragma unroll
  for (int j = 0; j < NQT; ++j)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float v = l_part[j][u];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      if (r == 0) red_l[warp * R + 8 * j + 2 * c + u] = v;
    }
  __syncthreads();
  float l_tot[NQT][2];
#pragma unroll
  for (int j = 0; j < NQT; ++j)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int qr = 8 * j + 2 * c + u;
      l_tot[j][u] = red_l[qr] + red_l[R + qr] + red_l[2 * R + qr] + red_l[3 * R + qr];
    }

  const bool final_out = (nsplit == 1);
  const int64_t part = (static_cast<int64_t>(b) * a.H + h) * a.target + split;
  const int dw0 = warp * Cfg::DW;
#pragma unroll
  for (int mt = 0; mt < Cfg::MT; ++mt)
#pragma unroll
    for (int j = 0; j < NQT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qr = 8 * j + 2 * c + (e & 1);
        if (qr >= R_real) continue;
        const int hi = e >> 1;
        int d;
        if constexpr (KV == KIND_BF16) {
          d = dw0 + 16 * mt + r + 8 * hi;
        } else {
          constexpr int EPT = Cfg::EPT;
          const int p = mt / (EPT / 2), mg = mt % (EPT / 2);
          d = dw0 + 8 * EPT * p + EPT * r + 2 * mg + hi;
        }
        if (final_out) {
          const float l = l_tot[j][e & 1];
          const int t = qr / a.G, g = qr % a.G;
          const int64_t oi = ((static_cast<int64_t>(b) * a.T + t) * a.Hq + h * a.G + g) * D + d;
          a.out[oi] = __float2bfloat16_rn(l > 0.f ? o[mt][j][e] / l : 0.f);
        } else {
          a.ws_acc[(part * R + qr) * D + d] = o[mt][j][e];
        }
      }
  if (r == 0) {
#pragma unroll
    for (int j = 0; j < NQT; ++j)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int qr = 8 * j + 2 * c + u;
        if (qr >= R_real || warp != 0) continue;
        if (final_out) {
          if (a.lse) {
            const int t = qr / a.G, g = qr % a.G;
            const float l = l_tot[j][u];
            a.lse[(static_cast<int64_t>(b) * a.T + t) * a.Hq + h * a.G + g] =
                l > 0.f ? (m_run[j][u] + log2f(l)) * kLn2 : -INFINITY;
          }
        } else {
          a.ws_ml[part * R + qr] = make_float2(m_run[j][u], l_tot[j][u]);
        }
      }
  }
}

// Launch of one instantiation; returns a cudaError_t.
struct DecodeLaunch {
  int smem_bytes;
  int nqt;
  const void* kernel;
};

template <int KK, int KV, int D, int NQT>
cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                          dim3 grid, cudaStream_t s) {
  using Cfg = DecodeCfg<KK, KV, D, NQT>;
  auto k = decode_kernel<KK, KV, D, NQT>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k<<<grid, 128, Cfg::SMEM, s>>>(tk, tv, a);
  return cudaGetLastError();
}

template <int KK, int KV, int D, int NQT>
int decode_ctas_per_sm() {
  using Cfg = DecodeCfg<KK, KV, D, NQT>;
  static int cached = 0;
  if (!cached) {
    auto k = decode_kernel<KK, KV, D, NQT>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, 128, Cfg::SMEM) != cudaSuccess || n < 1) n = 1;
    cached = n;
  }
  return cached;
}

// Per-profile entry points (defined in decode_<profile>.cu).
using DecodeFn = cudaError_t (*)(const nk_pool*, int layer, const DecodeArgs&, int nqt, dim3 grid,
                                 cudaStream_t);
using OccFn = int (*)(int D, int nqt);

template <int KK, int KV>
cudaError_t decode_dispatch(const nk_pool* p, int layer, const DecodeArgs& a, int nqt, dim3 grid,
                            cudaStream_t s) {
  const CUtensorMap& tk = p->tmap[layer * 2 + 0];
  const CUtensorMap& tv = p->tmap[layer * 2 + 1];
  const int D = p->desc.head_dim;
#define NK_CASE(DD, Q) \
  if (D == DD && nqt == Q) return launch_decode<KK, KV, DD, Q>(tk, tv, a, grid, s);
  NK_CASE(64, 1) NK_CASE(64, 2) NK_CASE(64, 4)
  NK_CASE(128, 1) NK_CASE(128, 2) NK_CASE(128, 4)
  NK_CASE(256, 1) NK_CASE(256, 2)
#undef NK_CASE
  return cudaErrorInvalidValue;
}

template <int KK, int KV>
int decode_occupancy(int D, int nqt) {
#define NK_CASE(DD, Q) \
  if (D == DD && nqt == Q) return decode_ctas_per_sm<KK, KV, DD, Q>();
  NK_CASE(64, 1) NK_CASE(64, 2) NK_CASE(64, 4)
  NK_CASE(128, 1) NK_CASE(128, 2) NK_CASE(128, 4)
  NK_CASE(256, 1) NK_CASE(256, 2)
#undef NK_CASE
  return 1;
}

cudaError_t decode_bf16(const nk_pool*, int, const DecodeArgs&, int, dim3, cudaStream_t);
cudaError_t decode_int8(const nk_pool*, int, const DecodeArgs&, int, dim3, cudaStream_t);
cudaError_t decode_fp8(const nk_pool*, int, const DecodeArgs&, int, dim3, cudaStream_t);
cudaError_t decode_nvfp4(const nk_pool*, int, const DecodeArgs&, int, dim3, cudaStream_t);
cudaError_t decode_k8v4(const nk_pool*, int, const DecodeArgs&, int, dim3, cudaStream_t);
int occupancy_bf16(int, int);
int occupancy_int8(int, int);
int occupancy_fp8(int, int);
int occupancy_nvfp4(int, int);
int occupancy_k8v4(int, int);

}  // namespace nk
