// decode.cuh -- split-K paged GQA decode / verify attention over the typed
// KV pool (kernel template; instantiated per profile in decode_*.cu).
//
// Contract ("Paged KV cache" maintainer design page, consumer view section):
// the consumer reads K/V pages in place through block_tables[table_rows[b]],
// translating logical block -> physical page once per page (never in the
// inner loop), with no gather-to-contiguous copy; a frontier may sit at any
// offset of the last page and bytes past it are never used.
//
// Work split.  A CTA owns one (row b, KV head h, page range).  The page
// ranges come from the device-side frontiers, so the host needs no lengths and
// the launch is graph-stable: with N_b = ceil(F_b / 64) pages, every CTA
// computes chunk = max(ceil(sum_b N_b / (target - B)), ceil(max_b N_b / 16)),
// row b gets ceil(N_b / chunk) splits (at most `target` in all: one wave; at
// most 16 per row), and CTA x of a head takes the x-th split.
//
// Warp roles.  The last warp is the producer: one lane stages page tiles (K
// codes, V codes, K / V scales of one (page, head)) into a ring of NSTAGE
// shared buffers with TMA / bulk copies, tracked by full / empty mbarriers.
// The consumers own 16-key slabs: slab p of every page is handled by one warp
// (D <= 128), or at D = 256 by a pair of warps that each own half of the head
// dims; a slab keeps its own online softmax, so the loop has no CTA-wide
// barrier:
//  QK:  partial S^T (16 keys x R query rows) over the warp's dims by
//       mma.m16n8k16 with the K tile as the A operand (ldmatrix of the raw
//       codes, exact conversion to f16 / bf16 in registers) and q as B; the
//       two halves are added through shared memory (same order in both
//       warps).  INT8-G64 group scales and FP8 row scales multiply fp32
//       partial sums; NVFP4 scales multiply the f16 operand (exact product).
//  softmax: base-2, per query row over the pair's keys, with a lazy reference
//       maximum that moves only when a score passes it by more than 2^8.
//  PV:  O^T (the warp's dims x R) += V^T P^T with P^T taken straight from the
//       S registers by movmatrix, V^T built in registers from the V tile
//       (ldmatrix.trans for bf16; byte gathers for 8-bit and 4-bit codes), V
//       scales folded in as f16 products.
// At the end the four pairs' (m, l, O) are combined in a fixed order, and the
// CTA writes unnormalised partials (m, l, acc) to the workspace, or the final
// out / lse when its row has a single split; merge_kernel, launched right
// behind, combines the splits.
#pragma once

#include "device.cuh"
#include "encode.cuh"
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
  // Fused append (nullptr: plain decode): the T new tokens of row b, bf16
  // [B][T][H][D], are encoded into positions F_b - T .. F_b - 1 of the
  // writable planes before the pages holding them are read.
  const __nv_bfloat16* k_new = nullptr;
  const __nv_bfloat16* v_new = nullptr;
  uint8_t* kc_w = nullptr;
  uint8_t* vc_w = nullptr;
  uint8_t* ks_w = nullptr;
  uint8_t* vs_w = nullptr;
  float softmax_scale;
  int B, T, Hq, H, G, L, M, C;
  int target;    // partial slots per (row, KV head) (= maxsplit); with nseg == 0 also the
                 // splits per head the chunking aims at, one CTA each
  int nseg = 0;  // > 0: pieces per head the chunking aims at, several per CTA (vdecode.cu)
  int ctas = 0;  // CTAs per KV head of the decode launch (read when nseg > 0)
  int head_major = 0;  // plane order
};

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
  // Head-dim split: at D = 256 with more than 8 query rows, or over INT8
  // pages (whose short contexts make the per-page latency count), the keys of
  // a 16-key slab are shared by a pair of warps, each owning half of the dims
  // (NH = 2); otherwise one warp per slab.
  static constexpr int NH = (D == 256 && (NQT > 1 || KK == KIND_INT8)) ? 2 : 1;
  static constexpr int NW = 4 * NH;              // consumer warps
  static constexpr int NCONS = 32 * NW;          // consumer threads
  static constexpr int THREADS = NCONS + 32;     // + 1 producer warp
  static constexpr int R = 8 * NQT;    // query rows (T * G) padded to n-tiles of 8
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
  // Ring depth: four stages of small tiles (several CTAs per SM), two of the
  // larger ones.
  static constexpr int NSTAGE = STAGE <= 16 * 1024 ? 4 : 2;
  static constexpr bool MMA_BF16 = (KK == KIND_BF16);
  static constexpr int Q_PITCH = D * 2 + 32;  // bytes per q row (padded against bank conflicts)
  // q fragments of a warp live in registers when they are few, else they are
  // read from shared memory (f16 / bf16 ready) at every k-step
  static constexpr bool Q_SMEM = (D / NH / 16) * NQT * 2 > 32 || NH == 2;
  // the final combine keeps one [R][D] fp32 slice per key slab group (4)
  static constexpr int COMB = 4 * R * D * 4;
  static constexpr int OFF_Q = align_up(NSTAGE * STAGE > COMB ? NSTAGE * STAGE : COMB, 128);
  static constexpr int OFF_X = OFF_Q + align_up(R * Q_PITCH, 128);   // partial-S exchange [2][NW][32][NQT*4]
  static constexpr int OFF_RED = OFF_X + (NH == 2 ? 2 * NW * 32 * NQT * 4 * 4 : 0);
  // per consumer warp: its 16 keys x its dims of V as f16 (quantized V), in
  // 64-dim blocks of 16 rows x 128 bytes, the source of the ldmatrix.trans
  // V^T fragments
  // (not for warp pairs launched two CTAs per SM: their register bound keeps
  // V^T in registers)
  static constexpr bool V_SMEM = KV != KIND_BF16 && (NH == 1 || (D / NH) * R / 32 > 32);
  static constexpr int VW_BYTES = V_SMEM ? 16 * (D / NH) * 2 : 0;  // 16 keys x the warp's dims, f16
  static constexpr int OFF_VW = align_up(OFF_RED + 10 * R * 4, 128);
  static constexpr int OFF_BAR = OFF_VW + NW * VW_BYTES;  // m, l per pair; M, L per row
  static constexpr int MISC_INTS = 32;
  static constexpr int SMEM = OFF_BAR + (2 * NSTAGE + 1) * 8 + MISC_INTS * 4 + 1024;  // + alignment slack
  static_assert(R * 32 * 12 <= OFF_Q, "merge weights of 32 splits fit below q");
  // CTAs per SM the register allocation aims at, from the O accumulators of
  // a warp ((D / NH) x R fp32 over 32 lanes).
  static constexpr int OREGS = (D / NH) * R / 32;
  static constexpr int MINB = NH == 2 ? (OREGS > 32 ? 1 : 2) : (OREGS > 32 ? 2 : 3);
};

// At most this many splits per (row, KV head): bounds the merge work of the
// last split.
constexpr int kMaxSplits = 32;

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

// Pages per split: with chunk = ceil(total / (target - B)) every row's
// ceil(N_b / chunk) splits add up to at most `target` (one wave of CTAs).
__host__ __device__ __forceinline__ int split_chunk(int total, int target, int B) {
  const int t = target - B > 1 ? target - B : 1;
  const int c = (total + t - 1) / t;
  return c < 1 ? 1 : c;
}

// The smallest chunk (at least ceil(maxp / kMaxSplits)) whose splits,
// max(1, ceil(N_b / chunk)) for every row, add up to at most `target`:
// split_chunk's value always qualifies, a bisection finds the least one, so
// the longest split is as short as one wave allows.
__device__ __forceinline__ int wave_chunk(const int* s_F, int B, int total, int maxp, int target) {
  const int floor_c = (maxp + kMaxSplits - 1) / kMaxSplits;
  int hi = max(split_chunk(total, target, B), floor_c);
  int lo = max(max(1, floor_c), (total + target - 1) / max(target, 1));
  if (lo > hi) lo = hi;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    int n = 0;
    for (int bb = 0; bb < B; ++bb) n += max(1, (((s_F[bb] + 63) >> 6) + mid - 1) / mid);
    if (n <= target) hi = mid;
    else lo = mid + 1;
  }
  return hi;
}

// Pages per piece when a CTA takes several pieces (a budget of nseg pieces
// per head): the pieces need not fit one wave, only each row's own slots.
__host__ __device__ __forceinline__ int seg_chunk(int total, int nseg) {
  const int c = (total + nseg - 1) / nseg;
  return c < 1 ? 1 : c;
}

// Pages per piece of the kernel that takes several pieces per CTA: about
// total / nseg while that leaves pieces of at least 64 pages; shorter pieces
// would cost more in per-piece hand-offs than they win in balance, so the
// plan falls back to one wave-filling split per CTA.
__device__ __forceinline__ int piece_chunk(const int* s_F, const DecodeArgs& a, int total, int maxp) {
  const int c = seg_chunk(total, a.nseg);
  if (c >= 64) return max(c, (maxp + kMaxSplits - 1) / kMaxSplits);
  return wave_chunk(s_F, a.B, total, maxp, min(a.ctas, a.target));
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Barrier of the consumer warps only (named barrier 1).
template <int NCONS>
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NCONS) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int KK, int KV, int D, int NQT>
__global__ void __launch_bounds__((DecodeCfg<KK, KV, D, NQT>::THREADS), (DecodeCfg<KK, KV, D, NQT>::MINB))
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  DecodeArgs a) {
  using Cfg = DecodeCfg<KK, KV, D, NQT>;
  constexpr int R = Cfg::R;
  constexpr int NSTAGE = Cfg::NSTAGE;
  constexpr int NH = Cfg::NH, NW = Cfg::NW, NCONS = Cfg::NCONS;
  constexpr int DH = D / NH;       // head dims of one consumer warp
  constexpr int KSW = DH / 16;     // k-steps of QK per warp
  constexpr int MTW = DH / 16;     // m-tiles of PV per warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs = smem + Cfg::OFF_Q;                                  // q rows [R][Q_PITCH]
  float* sx = reinterpret_cast<float*>(smem + Cfg::OFF_X);         // [2][8][32][NQT*4] partial S
  float* red_m = reinterpret_cast<float*>(smem + Cfg::OFF_RED);    // [4][R]
  float* red_l = red_m + 4 * R;                                     // [4][R]
  float* row_M = red_l + 4 * R;                                     // [R]
  float* row_L = row_M + R;                                         // [R]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* empty = full + NSTAGE;
  uint64_t* app = empty + NSTAGE;                           // fused append done (NW arrivals)
  int* s_flags = reinterpret_cast<int*>(app + 1);           // [0] abort
  int* s_F = s_flags + 4;                                   // [8] valid length per row
  int* s_row = s_flags + 12;                                // [8] table row per row
  float* s_qmax = reinterpret_cast<float*>(s_flags + 20);   // [8] per-warp max|q|

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  // consumers: keys [16 pair, +16), dims [half DH, +DH)
  const int pair = NH == 2 ? warp >> 1 : warp, half = NH == 2 ? warp & 1 : 0;
  const int h = blockIdx.y;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    mbar_init(app, NW);
    s_flags[0] = 0;
    s_flags[1] = 0;
    fence_barrier_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  // Launched with programmatic stream serialization: everything above overlaps
  // the previous kernel's tail; nothing it wrote is read before the wait.
  // The fused call's contract leaves only q and the new k / v to the previous
  // kernel (block tables, row map, frontiers and the pages of earlier tokens
  // are complete before it), so there the split plan and the page loads start
  // at once and only the consumers wait, before they read q, k or v and before
  // any global write.  The plain decode waits here (a separate append may have
  // just written its pages).
  const bool early = a.k_new != nullptr;
  if (!early) griddep_wait();
  griddep_launch_dependents();

  // ---- per-row lengths, loaded once in parallel ------------------------------
  if (tid < a.B) {
    const int F = a.frontiers[tid], row = a.table_rows[tid];
    const bool ok = F >= 0 && F <= a.L * 64 && row >= 0 && row < a.C && (a.k_new == nullptr || F >= a.T);
    if (!ok && blockIdx.x == 0 && h == 0) set_status(a.status, NK_STATUS_FRONTIER);
    s_F[tid] = ok ? F : 0;
    s_row[tid] = ok ? row : 0;
  }
  __syncthreads();

  // ---- which (row, split) this CTA owns --------------------------------------
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
      const int ns = max(1, (np + chunk - 1) / chunk);  // a row without keys still writes out / lse
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
  const int F = s_F[b];
  const int p0 = split * chunk;
  const int n = min(chunk, npages - p0);  // pages of this CTA (0 only for a row without keys)
  const bool fused = a.k_new != nullptr;
  const int app_lo = fused ? (F - a.T) >> 6 : 0x7fffffff;  // first page that receives new tokens
  const int R_real = a.T * a.G;

  // ---- producer warp: stage pages p0 .. p0+n-1 ---------------------------------
  if (warp == NW) {
    const int32_t* table = a.tables + static_cast<int64_t>(s_row[b]) * a.L + p0;
    int gnext = 0;
    bool app_seen = false;
    for (int i = 0; i < n; ++i) {
      if ((i & 31) == 0) gnext = (i + lane < n) ? table[i + lane] : 0;  // 32 table entries per load
      int g = __shfl_sync(0xffffffffu, gnext, i & 31);
      int stop = 0;
      if (lane == 0) {
        const int s = i % NSTAGE;
        if (p0 + i >= app_lo && !app_seen) {  // this page receives new tokens: wait for them
          app_seen = true;
          if (!mbar_wait_bounded(app, 0, a.status)) stop = 1;
        }
        if (stop || (i >= NSTAGE && !mbar_wait_bounded(&empty[s], ((i / NSTAGE) - 1) & 1, a.status))) {
          s_flags[0] = 1;
          stop = 1;
        } else {
          if (g < 0 || g >= a.M) {  // never copy from outside the pool
            set_status(a.status, NK_STATUS_PAGE_RANGE);
            g = 0;                  // the row's result is then undefined
          }
          uint8_t* st = smem + s * Cfg::STAGE;
          const int y = static_cast<int>(tile_row(g, h, a.H, a.M, a.head_major));
          mbar_arrive_expect_tx(&full[s], Cfg::TX_BYTES);
#pragma unroll
          for (int j = 0; j < Cfg::KCB / Cfg::K_RB; ++j)
            tma_load_2d(st + j * 64 * Cfg::K_RB, &tmk, j * Cfg::K_RB, y, &full[s]);
#pragma unroll
          for (int j = 0; j < Cfg::VCB / Cfg::V_RB; ++j)
            tma_load_2d(st + Cfg::OFF_V + j * 64 * Cfg::V_RB, &tmv, j * Cfg::V_RB, y, &full[s]);
          if constexpr (Cfg::KS_TILE > 0) {
            bulk_load(st + Cfg::OFF_KS, a.ks + static_cast<int64_t>(y) * Cfg::KSB, Cfg::KS_TILE, &full[s]);
            bulk_load(st + Cfg::OFF_VS, a.vs + static_cast<int64_t>(y) * Cfg::VSB, Cfg::VS_TILE, &full[s]);
          }
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) break;
    }
    return;  // the copies complete into the shared memory of the still-running CTA
  }

  if (early) {
    // the q rows of this (row, KV head) and its new k / v rows into L2 while the
    // previous kernel finishes; they are read right after the wait
    if (tid < a.T) {
      const int64_t bt = static_cast<int64_t>(b) * a.T + tid;
      prefetch_l2(a.q + (bt * a.Hq + h * a.G) * D, a.G * D * 2);
      prefetch_l2(a.k_new + (bt * a.H + h) * D, D * 2);
      prefetch_l2(a.v_new + (bt * a.H + h) * D, D * 2);
    }
    griddep_wait();  // consumers: q, k, v and all writes come after the previous kernel
  }

  // ---- fused append: the new tokens whose pages this CTA reads ------------------
  // One consumer warp per token encodes its K and V rows of head h into the
  // pool, then orders those generic-proxy stores before the producer's TMA
  // reads of the same bytes (fence.proxy.async + the app mbarrier).
  if (fused) {
    constexpr int KCBW = code_row_bytes<KK>(D), VCBW = code_row_bytes<KV>(D);
    constexpr int KSBW = scale_row_bytes<KK>(D), VSBW = scale_row_bytes<KV>(D);
    const int32_t* trow = a.tables + static_cast<int64_t>(s_row[b]) * a.L;
    for (int t = warp; t < a.T; t += NW) {
      const int pos = F - a.T + t;
      const int pg = pos >> 6;
      if (pg < p0 || pg >= p0 + n) continue;
      const int g = trow[pg];
      if (g < 0 || g >= a.M) {
        if (lane == 0) set_status(a.status, NK_STATUS_PAGE_RANGE);
        continue;
      }
      const int64_t token_row = tile_row(g, h, a.H, a.M, a.head_major) + (pos & 63);
      const int64_t src = ((static_cast<int64_t>(b) * a.T + t) * a.H + h) * D;
      encode_row<KK, D>(a.k_new + src, a.kc_w + token_row * KCBW, a.ks_w ? a.ks_w + token_row * KSBW : nullptr, lane);
      encode_row<KV, D>(a.v_new + src, a.vc_w + token_row * VCBW, a.vs_w ? a.vs_w + token_row * VSBW : nullptr, lane);
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(app);
  }

  // ---- q rows to shared memory (16-byte loads) and the f16 prescale --------------
  // Row qr = t * G + g of this CTA is q[b][t][h * G + g][:]; the G rows of one
  // token are contiguous.  Padded rows (qr >= T * G) are zero.  Quantized
  // profiles run the MMAs in f16: q is scaled by 2^e so that max|q| * 2^e lies
  // in [2^14, 2^15) (exact for every element above max|q| * 2^-31), and the
  // scores divide 2^e back out.
  float mx = 0.f;
  {
    constexpr int V8 = D / 8;  // uint4 per row
    for (int i = tid; i < R * V8; i += NCONS) {
      const int qr = i / V8, col = i % V8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (qr < R_real) {
        const int t = qr / a.G, g = qr % a.G;
        v = *reinterpret_cast<const uint4*>(
            a.q + ((static_cast<int64_t>(b) * a.T + t) * a.Hq + h * a.G + g) * D + col * 8);
      }
      *reinterpret_cast<uint4*>(qs + qr * Cfg::Q_PITCH + col * 16) = v;
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
      for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fabsf(__bfloat162float(e[k])));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) s_qmax[warp] = mx;
  }
  consumer_sync<NCONS>();
#pragma unroll
  for (int w = 0; w < NW; ++w) mx = fmaxf(mx, s_qmax[w]);
  float qscale_log2 = 0.f, qf_mul = 1.f;
  if constexpr (!Cfg::MMA_BF16) {
    int ex = 0;
    if (mx > 0.f) frexpf(mx, &ex);
    const int e = mx > 0.f ? min(15 - ex, 100) : 0;  // 2^e stays finite in fp32
    qf_mul = ldexpf(1.f, e);
    qscale_log2 = static_cast<float>(e);
  }
  const float sc = a.softmax_scale * kLog2e * exp2f(-qscale_log2);

  // q fragments of this warp's k-steps (global k-step half * KSW + s), in
  // registers, or converted in place in shared memory when Q_SMEM
  if constexpr (Cfg::Q_SMEM && !Cfg::MMA_BF16) {
    for (int i2 = tid; i2 < R * D / 2; i2 += NCONS) {
      const int qr = i2 / (D / 2), col = i2 % (D / 2);
      uint32_t* p = reinterpret_cast<uint32_t*>(qs + qr * Cfg::Q_PITCH + col * 4);
      const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(p);
      *p = pack_f16x2(__low2float(v) * qf_mul, __high2float(v) * qf_mul);
    }
    consumer_sync<NCONS>();
  }
  auto qfrag = [&](int s, int j, uint32_t& b0, uint32_t& b1) {
    const uint8_t* row = qs + (8 * j + r) * Cfg::Q_PITCH;
    const int sg = half * KSW + s;
    if constexpr (KK == KIND_BF16) {
      b0 = *reinterpret_cast<const uint32_t*>(row + 2 * q_dim<KK>(sg, 0, c));
      b1 = *reinterpret_cast<const uint32_t*>(row + 2 * q_dim<KK>(sg, 2, c));
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(row + 2 * q_dim<KK>(sg, 0, c));
      b0 = v.x;
      b1 = v.y;
    }
  };
  uint32_t qreg[Cfg::Q_SMEM ? 1 : KSW][Cfg::Q_SMEM ? 1 : NQT][2];
  if constexpr (!Cfg::Q_SMEM) {
#pragma unroll
    for (int s = 0; s < KSW; ++s)
#pragma unroll
      for (int j = 0; j < NQT; ++j) {
        const uint8_t* row = qs + (8 * j + r) * Cfg::Q_PITCH;
        const int sg = half * KSW + s;
        if constexpr (Cfg::MMA_BF16) {
          qfrag(s, j, qreg[s][j][0], qreg[s][j][1]);
        } else {
          float v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            v[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(row + 2 * q_dim<KK>(sg, i, c))) * qf_mul;
          qreg[s][j][0] = pack_f16x2(v[0], v[1]);
          qreg[s][j][1] = pack_f16x2(v[2], v[3]);
        }
      }
  }
  // B operand of k-step s, n-tile j
  auto qb = [&](int s, int j, uint32_t& b0, uint32_t& b1) {
    if constexpr (Cfg::Q_SMEM) qfrag(s, j, b0, b1);
    else b0 = qreg[s][j][0], b1 = qreg[s][j][1];
  };

  // ---- running state -----------------------------------------------------------
  // nm: minus the row's reference maximum (0 before the row's first key),
  // folded into the score scaling as one FFMA per score
  float nm[NQT][2], l_part[NQT][2];
  float o[MTW][NQT][4];
  // INT8-G64 / FP8-row V: the values are f16 products code * (s 2^k_run), with
  // k_run <= 0 the lift of the largest value scale this warp has read
  // (v_lift): 0 for every V below 2^7 * 127 (INT8) or 2^7 * 448 (FP8), less
  // above, so that no product overflows f16 whatever the magnitude of V.  O
  // carries 2^k_run and is rescaled when it drops; the combine removes it.
  constexpr bool V_LIFT = KV == KIND_INT8 || KV == KIND_FP8;
  int k_run = 0;
#pragma unroll
  for (int j = 0; j < NQT; ++j) {
    nm[j][0] = nm[j][1] = 0.f;
    l_part[j][0] = l_part[j][1] = 0.f;
  }
#pragma unroll
  for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
    for (int j = 0; j < NQT; ++j) o[mt][j][0] = o[mt][j][1] = o[mt][j][2] = o[mt][j][3] = 0.f;

  // query row qr may see keys <= F - T + qr / G (and < F)
  int lim[NQT][2];
#pragma unroll
  for (int j = 0; j < NQT; ++j)
#pragma unroll
    for (int u = 0; u < 2; ++u) lim[j][u] = min(F - a.T + (8 * j + 2 * c + u) / a.G, F - 1);

  const int kr0 = 16 * pair + r, kr1 = kr0 + 8;                        // keys of this thread's S rows
  const int krow_ld = 16 * pair + (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row of this lane
  const int kk0 = 16 * pair + 2 * c;                                   // first PV key of this thread
  const uint32_t pair_bar = 2 + pair;                                  // named barrier of the warp pair

  bool aborted = false;
  int i = 0;
  for (; i < n; ++i) {
    const int s = i % NSTAGE;
    const uint8_t* st = smem + s * Cfg::STAGE;
    const uint32_t kbase = smem_u32(st);
    const uint32_t vbase = smem_u32(st + Cfg::OFF_V);
    if (!mbar_wait_bounded(&full[s], (i / NSTAGE) & 1, a.status)) {
      aborted = true;
      break;
    }
    const int key0 = (p0 + i) * 64;

    // V lift: the largest scale of this warp's 16 keys below the frontier
    // (lane: key 16 pair + lane % 16; INT8 groups of the warp's dims split by
    // lane / 16), across the warp
    int knew = k_run;
    if constexpr (V_LIFT) {
      const uint16_t* vsp = reinterpret_cast<const uint16_t*>(st + Cfg::OFF_VS);
      const int vk = 16 * pair + (lane & 15);
      float smax = 0.f;
      if (key0 + vk < F) {
        if constexpr (KV == KIND_INT8) {
          constexpr int GW = DH >= 64 ? DH / 64 : 1;
#pragma unroll
          for (int gi = lane >> 4; gi < GW; gi += 2)
            smax = fmaxf(smax, __half2float(__ushort_as_half(vsp[vk * (Cfg::VSB / 2) + (half * DH) / 64 + gi])));
        } else {
          smax = __half2float(__ushort_as_half(vsp[vk]));
        }
      }
      knew = v_lift(__reduce_max_sync(0xffffffffu, __float_as_uint(smax)), k_run);
    }

    // ---------------- QK: partial S^T over this warp's head dims ------------------
    float S[NQT][4];
#pragma unroll
    for (int j = 0; j < NQT; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
    const uint8_t* ks_tile = st + Cfg::OFF_KS;
    if constexpr (KK == KIND_BF16) {
#pragma unroll
      for (int s16 = 0; s16 < KSW; ++s16) {
        const int col = (2 * (half * KSW + s16) + (lane >> 4)) * 16;
        const uint32_t addr = kbase + (col / 128) * (64 * 128) + swz<128>(krow_ld, col % 128);
        uint32_t A[4];
        ldsm_x4(addr, A[0], A[1], A[2], A[3]);
#pragma unroll
        for (int j = 0; j < NQT; ++j) {
          uint32_t b0, b1;
          qb(s16, j, b0, b1);
          mma16816<true>(S[j], A, b0, b1);
        }
      }
    } else if constexpr (KK == KIND_NVFP4) {
      constexpr int RB = Cfg::K_RB;
      constexpr int NCW = Cfg::KCB / 16 / NH;  // 16-byte chunks (32 dims) of this warp
#pragma unroll
      for (int cw = 0; cw < NCW; cw += 2) {
        const int cc0 = half * NCW + cw;
        const int col = (cc0 + (NCW > 1 ? (lane >> 4) : 0)) * 16;
        const uint32_t addr = kbase + (col / RB) * (64 * RB) + swz<RB>(krow_ld, col % RB);
        uint32_t d[4];
        ldsm_x4(addr, d[0], d[1], d[2], d[3]);
#pragma unroll
        for (int u = 0; u < (NCW > 1 ? 2 : 1); ++u) {  // chunk cc0+u: regs d[2u] (key r), d[2u+1] (key r+8)
          const int cc = cc0 + u;
          const int blk = 2 * cc + (c >> 1);
          const __half s0 = __ushort_as_half(static_cast<uint16_t>(
              e4m3x2_to_f16x2(ks_tile[kr0 * Cfg::KSB + blk]) & 0xFFFFu));
          const __half s1 = __ushort_as_half(static_cast<uint16_t>(
              e4m3x2_to_f16x2(ks_tile[kr1 * Cfg::KSB + blk]) & 0xFFFFu));
          const uint32_t sc0 = pack_h2(s0, s0), sc1 = pack_h2(s1, s1);
          const uint32_t w0 = d[2 * u], w1 = d[2 * u + 1];
          const uint32_t A0[4] = {hmul2_u32(e2m1x2_byte_to_f16x2<0>(w0), sc0), hmul2_u32(e2m1x2_byte_to_f16x2<0>(w1), sc1),
                                  hmul2_u32(e2m1x2_byte_to_f16x2<1>(w0), sc0), hmul2_u32(e2m1x2_byte_to_f16x2<1>(w1), sc1)};
          const uint32_t A1[4] = {hmul2_u32(e2m1x2_byte_to_f16x2<2>(w0), sc0), hmul2_u32(e2m1x2_byte_to_f16x2<2>(w1), sc1),
                                  hmul2_u32(e2m1x2_byte_to_f16x2<3>(w0), sc0), hmul2_u32(e2m1x2_byte_to_f16x2<3>(w1), sc1)};
          const int sl = 2 * (cw + u);  // local k-steps of this chunk
#pragma unroll
          for (int j = 0; j < NQT; ++j) {
            uint32_t b0, b1, c0, c1;
            qb(sl, j, b0, b1);
            qb(sl + 1, j, c0, c1);
            mma16816<false>(S[j], A0, b0, b1);
            mma16816<false>(S[j], A1, c0, c1);
          }
        }
      }
    } else {  // INT8 / FP8: 16 dims per 16-byte chunk
      constexpr int RB = Cfg::K_RB;
      constexpr int NCW = Cfg::KCB / 16 / NH;  // chunks of this warp (even)
      constexpr bool LOCAL_GROUPS = (KK == KIND_INT8) && (DH >= 64);
      float Sg[NQT][4];
#pragma unroll
      for (int cw = 0; cw < NCW; cw += 2) {
        if constexpr (LOCAL_GROUPS) {
          if ((cw & 3) == 0) {
#pragma unroll
            for (int j = 0; j < NQT; ++j) Sg[j][0] = Sg[j][1] = Sg[j][2] = Sg[j][3] = 0.f;
          }
        }
        const int col = (half * NCW + cw + (lane >> 4)) * 16;
        const uint32_t addr = kbase + (col / RB) * (64 * RB) + swz<RB>(krow_ld, col % RB);
        uint32_t d[4];
        ldsm_x4(addr, d[0], d[1], d[2], d[3]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t A[4] = {cvt_pair<KK, false>(d[2 * u]), cvt_pair<KK, false>(d[2 * u + 1]),
                                 cvt_pair<KK, true>(d[2 * u]), cvt_pair<KK, true>(d[2 * u + 1])};
#pragma unroll
          for (int j = 0; j < NQT; ++j) {
            uint32_t b0, b1;
            qb(cw + u, j, b0, b1);
            if constexpr (LOCAL_GROUPS) mma16816<false>(Sg[j], A, b0, b1);
            else mma16816<false>(S[j], A, b0, b1);
          }
        }
        if constexpr (LOCAL_GROUPS) {
          if ((cw & 3) == 2) {  // end of a 64-dim group: apply its scale
            const int grp = (half * NCW + cw) >> 2;
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
    }

    // ---------------- full S: add the partner warp's half (same order in both) ------
    if constexpr (NH == 2) {
      float* mine = sx + (((i & 1) * NW + warp) * 32 + lane) * (NQT * 4);
      const float* other = sx + (((i & 1) * NW + (warp ^ 1)) * 32 + lane) * (NQT * 4);
#pragma unroll
      for (int j = 0; j < NQT; ++j)
        *reinterpret_cast<float4*>(mine + 4 * j) = make_float4(S[j][0], S[j][1], S[j][2], S[j][3]);
      asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
#pragma unroll
      for (int j = 0; j < NQT; ++j) {
        const float4 v = *reinterpret_cast<const float4*>(other + 4 * j);
        if (half == 0) {
          S[j][0] += v.x; S[j][1] += v.y; S[j][2] += v.z; S[j][3] += v.w;
        } else {
          S[j][0] = v.x + S[j][0]; S[j][1] = v.y + S[j][1]; S[j][2] = v.z + S[j][2]; S[j][3] = v.w + S[j][3];
        }
      }
    }
    if constexpr ((KK == KIND_INT8 && DH < 64) || KK == KIND_FP8) {
      // FP8 row scale, or the single INT8 group shared by both halves
      const float g0 = __half2float(*reinterpret_cast<const __half*>(ks_tile + kr0 * Cfg::KSB));
      const float g1 = __half2float(*reinterpret_cast<const __half*>(ks_tile + kr1 * Cfg::KSB));
#pragma unroll
      for (int j = 0; j < NQT; ++j) {
        S[j][0] *= g0;
        S[j][1] *= g0;
        S[j][2] *= g1;
        S[j][3] *= g1;
      }
    }

    // ---------------- scores, masking, online softmax (this pair's keys) ---------------
    const int kg0 = key0 + kr0, kg1 = key0 + kr1;
    float alpha[NQT][2];
    bool rescale = false;
    // Lazy rescale: a row's reference maximum moves only when one of its
    // scores passes it by more than 2^8 (log2 units), so p <= 2^8 (exact in
    // the f16 / bf16 operands, harmless to the fp32 accumulators); a warp
    // vote on the thread-local maxima skips the cross-lane reduction of every
    // other page.  S becomes t = s - reference.  The first page always takes
    // the exact maximum: a row's visible keys are a prefix of the keys, so a
    // row with no visible key on the warp's first page has none later.
    const bool first = (i == 0);
    float vloc[NQT][2];
    bool need = first;
#pragma unroll
    for (int j = 0; j < NQT; ++j) {
      S[j][0] = kg0 <= lim[j][0] ? fmaf(S[j][0], sc, nm[j][0]) : -INFINITY;
      S[j][1] = kg0 <= lim[j][1] ? fmaf(S[j][1], sc, nm[j][1]) : -INFINITY;
      S[j][2] = kg1 <= lim[j][0] ? fmaf(S[j][2], sc, nm[j][0]) : -INFINITY;
      S[j][3] = kg1 <= lim[j][1] ? fmaf(S[j][3], sc, nm[j][1]) : -INFINITY;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        vloc[j][u] = fmaxf(S[j][u], S[j][2 + u]);
        need |= vloc[j][u] > 8.f;
      }
    }
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int j = 0; j < NQT; ++j)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float v = vloc[j][u];
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
          // first page: the reference becomes the row's maximum (l and O are
          // still 0); later: it moves up by the excess, if any
          const float shift = first ? (v == -INFINITY ? 0.f : v) : fmaxf(v, 0.f);
          alpha[j][u] = first ? 0.f : ex2(-shift);
          rescale |= shift > 0.f;
          nm[j][u] -= shift;
          S[j][u] = ex2(S[j][u] - shift);
          S[j][2 + u] = ex2(S[j][2 + u] - shift);
          l_part[j][u] = l_part[j][u] * alpha[j][u] + S[j][u] + S[j][2 + u];
        }
    } else {
#pragma unroll
      for (int j = 0; j < NQT; ++j)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          alpha[j][u] = 1.f;
          S[j][u] = ex2(S[j][u]);
          S[j][2 + u] = ex2(S[j][2 + u]);
          l_part[j][u] += S[j][u] + S[j][2 + u];
        }
    }
    if (__any_sync(0xffffffffu, rescale) || knew != k_run) {
      const float kf = pow2i(knew - k_run);
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
        for (int j = 0; j < NQT; ++j) {
          o[mt][j][0] *= alpha[j][0] * kf;
          o[mt][j][1] *= alpha[j][1] * kf;
          o[mt][j][2] *= alpha[j][0] * kf;
          o[mt][j][3] *= alpha[j][1] * kf;
        }
    }
    k_run = knew;
    const uint32_t lift2 = static_cast<uint32_t>(k_run + 15) * 0x04000400u;  // f16x2 (2^k_run, 2^k_run)
    // P^T as the B operand of PV, straight from registers: (key r, rows 2c,2c+1)
    // transposed by movmatrix gives (row r, keys 2c, 2c+1).
    uint32_t pb[Cfg::MMA_BF16 ? 2 : 1][NQT][2];
#pragma unroll
    for (int j = 0; j < NQT; ++j) {
      if constexpr (Cfg::MMA_BF16) {
        // bf16 P as hi + lo parts (about 16 significant bits)
        const __nv_bfloat162 hi0 = __floats2bfloat162_rn(S[j][0], S[j][1]);
        const __nv_bfloat162 hi1 = __floats2bfloat162_rn(S[j][2], S[j][3]);
        const __nv_bfloat162 lo0 = __floats2bfloat162_rn(S[j][0] - __low2float(hi0), S[j][1] - __high2float(hi0));
        const __nv_bfloat162 lo1 = __floats2bfloat162_rn(S[j][2] - __low2float(hi1), S[j][3] - __high2float(hi1));
        pb[0][j][0] = movm_t(*reinterpret_cast<const uint32_t*>(&hi0));
        pb[0][j][1] = movm_t(*reinterpret_cast<const uint32_t*>(&hi1));
        pb[Cfg::MMA_BF16 ? 1 : 0][j][0] = movm_t(*reinterpret_cast<const uint32_t*>(&lo0));
        pb[Cfg::MMA_BF16 ? 1 : 0][j][1] = movm_t(*reinterpret_cast<const uint32_t*>(&lo1));
      } else {
        pb[0][j][0] = movm_t(pack_f16x2(S[j][0], S[j][1]));
        pb[0][j][1] = movm_t(pack_f16x2(S[j][2], S[j][3]));
      }
    }

    // ---------------- PV: O^T(this warp's dims x R) += V^T P^T over the pair's keys ------
    const int kvalid = F - key0;  // keys >= kvalid of this page are past the frontier
    uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
    if (kvalid < 64) {
      mlo = (kk0 < kvalid ? 0x0000FFFFu : 0u) | (kk0 + 1 < kvalid ? 0xFFFF0000u : 0u);
      mhi = (kk0 + 8 < kvalid ? 0x0000FFFFu : 0u) | (kk0 + 9 < kvalid ? 0xFFFF0000u : 0u);
    }
    if constexpr (KV == KIND_BF16) {
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt) {
        const int key = 16 * pair + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int col = (half * DH + 16 * mt + 8 * ((lane >> 3) & 1)) * 2;
        const uint32_t addr = vbase + (col / 128) * (64 * 128) + swz<128>(key, col % 128);
        uint32_t A[4];
        ldsm_x4_t(addr, A[0], A[1], A[2], A[3]);
        A[0] &= mlo;
        A[1] &= mlo;
        A[2] &= mhi;
        A[3] &= mhi;
#pragma unroll
        for (int j = 0; j < NQT; ++j) {
          mma16816<true>(o[mt][j], A, pb[0][j][0], pb[0][j][1]);
          mma16816<true>(o[mt][j], A, pb[Cfg::MMA_BF16 ? 1 : 0][j][0], pb[Cfg::MMA_BF16 ? 1 : 0][j][1]);
        }
      }
    } else if constexpr (Cfg::V_SMEM) {
      // The warp converts its 16 keys x DH dims of V to f16 into its own
      // scratch (64-dim blocks of 16 key rows x 128 bytes, 128-byte swizzle),
      // with the scales applied (NVFP4: an exact product; INT8 / FP8: the f16
      // product) and keys past the frontier zeroed; ldmatrix.trans then gives
      // the V^T fragments, as for BF16 pages.  Lane: key slab row kr = lane &
      // 15, dims [32 dh, 32 dh + 32) of every 64-dim block, dh = lane >> 4.
      constexpr int RB = Cfg::V_RB;
      const uint8_t* vs_tile = st + Cfg::OFF_VS;
      const uint8_t* vtile = st + Cfg::OFF_V;
      uint8_t* vw = smem + Cfg::OFF_VW + warp * Cfg::VW_BYTES;
      const int kr = lane & 15, dh = lane >> 4;
      const int vkey = 16 * pair + kr;              // key of the page this lane converts
      const bool vlive = key0 + vkey < F;           // keys at or past the frontier are zero
      __syncwarp();  // the previous page's fragments have been read
#pragma unroll
      for (int q64 = 0; q64 < DH / 64; ++q64) {
        uint8_t* blk = vw + q64 * (16 * 128);
        const int d0 = half * DH + 64 * q64 + 32 * dh;  // first of this lane's 32 dims
        if constexpr (KV == KIND_NVFP4) {
          const int colb = d0 / 2;  // 16 code bytes, two scale bytes
          const uint4 w = *reinterpret_cast<const uint4*>(vtile + (colb / RB) * (64 * RB) + swz<RB>(vkey, colb % RB));
          // a key past the frontier gets zero scales: its E2M1 codes are
          // finite, so every product is 0 (stale scale bytes never enter)
          const uint32_t s2 =
              vlive ? e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(vs_tile + vkey * Cfg::VSB + d0 / 16)) : 0u;
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int sub = 0; sub < 2; ++sub) {  // 16 dims, one scale group
            const uint32_t sq = __byte_perm(s2, 0, sub ? 0x3232 : 0x1010);
            uint32_t hv[8];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              hv[4 * q + 0] = hmul2_u32(e2m1x2_byte_to_f16x2<0>(wv[2 * sub + q]), sq);
              hv[4 * q + 1] = hmul2_u32(e2m1x2_byte_to_f16x2<1>(wv[2 * sub + q]), sq);
              hv[4 * q + 2] = hmul2_u32(e2m1x2_byte_to_f16x2<2>(wv[2 * sub + q]), sq);
              hv[4 * q + 3] = hmul2_u32(e2m1x2_byte_to_f16x2<3>(wv[2 * sub + q]), sq);
            }
#pragma unroll
            for (int k = 0; k < 2; ++k)
              *reinterpret_cast<uint4*>(blk + swz<128>(kr, 64 * dh + 32 * sub + 16 * k)) =
                  make_uint4(hv[4 * k], hv[4 * k + 1], hv[4 * k + 2], hv[4 * k + 3]);
          }
        } else {  // INT8 / FP8: 16 code bytes per 16 dims
          const uint16_t* sp = reinterpret_cast<const uint16_t*>(vs_tile);
          const uint32_t s1 = KV == KIND_INT8 ? sp[vkey * (Cfg::VSB / 2) + d0 / 64] : sp[vkey];
          // INT8 codes are finite, so a zero scale zeroes a key past the
          // frontier; FP8 codes may encode NaN there and are selected away
          const uint32_t s2 = KV == KIND_INT8 && !vlive ? 0u : hmul2_u32(s1 | (s1 << 16), lift2);
#pragma unroll
          for (int sub = 0; sub < 2; ++sub) {
            const int dd = d0 + 16 * sub;
            const uint4 w = *reinterpret_cast<const uint4*>(vtile + (dd / RB) * (64 * RB) + swz<RB>(vkey, dd % RB));
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
            uint32_t hv[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if constexpr (KV == KIND_INT8) {
                hv[2 * q] = hmul2_u32(s8pair_to_f16x2(__byte_perm(wv[q], 0, 0x1100)), s2);
                hv[2 * q + 1] = hmul2_u32(s8pair_to_f16x2(__byte_perm(wv[q], 0, 0x3322)), s2);
              } else {
                hv[2 * q] = hmul2_u32(e4m3x2_to_f16x2(static_cast<uint16_t>(wv[q] & 0xFFFFu)), s2);
                hv[2 * q + 1] = hmul2_u32(e4m3x2_to_f16x2(static_cast<uint16_t>(wv[q] >> 16)), s2);
              }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint4 v = KV == KIND_INT8 || vlive ? make_uint4(hv[4 * k], hv[4 * k + 1], hv[4 * k + 2], hv[4 * k + 3])
                                                       : make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(blk + swz<128>(kr, 64 * dh + 32 * sub + 16 * k)) = v;
            }
          }
        }
      }
      __syncwarp();
#pragma unroll
      for (int q64 = 0; q64 < DH / 64; ++q64) {
#pragma unroll
        for (int mt4 = 0; mt4 < 4; ++mt4) {  // the block's four 16-dim m-tiles
          const int key = (lane & 7) + ((lane >> 4) & 1) * 8;
          const int col = (16 * mt4 + 8 * ((lane >> 3) & 1)) * 2;
          uint32_t A[4];
          ldsm_x4_t(smem_u32(vw + q64 * (16 * 128)) + swz<128>(key, col), A[0], A[1], A[2], A[3]);
#pragma unroll
          for (int j = 0; j < NQT; ++j) mma16816<false>(o[4 * q64 + mt4][j], A, pb[0][j][0], pb[0][j][1]);
        }
      }
    } else {  // head_dim 256: V^T fragments built in registers (byte gathers, prmt)
      constexpr int RB = Cfg::V_RB;
      const int keys[4] = {kk0, kk0 + 1, kk0 + 8, kk0 + 9};
      const uint8_t* vs_tile = st + Cfg::OFF_VS;
      const uint8_t* vtile = st + Cfg::OFF_V;
#pragma unroll
      for (int p = 0; p < DH / 32; ++p) {  // groups of 32 dims = 2 m-tiles
        const int dthr = half * DH + 32 * p + 4 * r;  // first dim of this thread in the group
        uint32_t pair_lo[4], pair_hi[4];
        if constexpr (KV == KIND_NVFP4) {
          uint32_t f[4][2];
#pragma unroll
          for (int kx = 0; kx < 4; ++kx) {
            const int colb = dthr / 2;
            const uint32_t wv = *reinterpret_cast<const uint16_t*>(vtile + (colb / RB) * (64 * RB) +
                                                                   swz<RB>(keys[kx], colb % RB));
            const __half sv = __ushort_as_half(static_cast<uint16_t>(
                e4m3x2_to_f16x2(vs_tile[keys[kx] * Cfg::VSB + dthr / 16]) & 0xFFFFu));
            const uint32_t s2 = pack_h2(sv, sv);
            f[kx][0] = hmul2_u32(e2m1x2_byte_to_f16x2<0>(wv), s2);
            f[kx][1] = hmul2_u32(e2m1x2_byte_to_f16x2<1>(wv), s2);
          }
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            pair_lo[2 * e2] = __byte_perm(f[0][e2], f[1][e2], 0x5410);
            pair_lo[2 * e2 + 1] = __byte_perm(f[0][e2], f[1][e2], 0x7632);
            pair_hi[2 * e2] = __byte_perm(f[2][e2], f[3][e2], 0x5410);
            pair_hi[2 * e2 + 1] = __byte_perm(f[2][e2], f[3][e2], 0x7632);
          }
        } else {
          uint32_t wv[4];
#pragma unroll
          for (int kx = 0; kx < 4; ++kx)
            wv[kx] = *reinterpret_cast<const uint32_t*>(vtile + (dthr / RB) * (64 * RB) +
                                                        swz<RB>(keys[kx], dthr % RB));
          uint32_t slo, shi;  // (s_key0, s_key1), (s_key8, s_key9) as f16x2
          const uint16_t* sp = reinterpret_cast<const uint16_t*>(vs_tile);
          if constexpr (KV == KIND_INT8) {
            const int grp = dthr / 64;
            slo = sp[keys[0] * (Cfg::VSB / 2) + grp] | (uint32_t(sp[keys[1] * (Cfg::VSB / 2) + grp]) << 16);
            shi = sp[keys[2] * (Cfg::VSB / 2) + grp] | (uint32_t(sp[keys[3] * (Cfg::VSB / 2) + grp]) << 16);
          } else {
            slo = sp[keys[0]] | (uint32_t(sp[keys[1]]) << 16);
            shi = sp[keys[2]] | (uint32_t(sp[keys[3]]) << 16);
          }
          slo = hmul2_u32(slo, lift2);
          shi = hmul2_u32(shi, lift2);
          if constexpr (KV == KIND_INT8) {  // finite codes: zero scales zero the keys past the frontier
            slo &= mlo;
            shi &= mhi;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
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
        for (int mg = 0; mg < 2; ++mg) {
          // keys past the frontier are zero (INT8: through their scales)
          const uint32_t ml = KV == KIND_INT8 ? 0xFFFFFFFFu : mlo, mh = KV == KIND_INT8 ? 0xFFFFFFFFu : mhi;
          const uint32_t A[4] = {pair_lo[2 * mg] & ml, pair_lo[2 * mg + 1] & ml,
                                 pair_hi[2 * mg] & mh, pair_hi[2 * mg + 1] & mh};
#pragma unroll
          for (int j = 0; j < NQT; ++j) mma16816<false>(o[2 * p + mg][j], A, pb[0][j][0], pb[0][j][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- combine the four pairs (fixed order), write partials or the output -----------
  // Both warps of a pair hold the same (m, l); each holds O for its own dims.
  // m is the reference maximum, -inf for a row that saw no key (l = 0; a row
  // that saw one has l >= 1: its maximum key had p = 1 when it was taken).
  float m_run[NQT][2];
#pragma unroll
  for (int j = 0; j < NQT; ++j)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float v = l_part[j][u];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      m_run[j][u] = v > 0.f ? -nm[j][u] : -INFINITY;
      if (r == 0 && half == 0) {
        red_m[pair * R + 8 * j + 2 * c + u] = m_run[j][u];
        red_l[pair * R + 8 * j + 2 * c + u] = v;
      }
    }
  if (aborted && lane == 0) s_flags[0] = 1;
  consumer_sync<NCONS>();
  if (s_flags[0]) {
    // drain copies that may still be in flight, then leave without results
    if (tid == 0)
      for (int k = i; k < min(n, i + NSTAGE); ++k)
        mbar_wait_bounded(&full[k % NSTAGE], (k / NSTAGE) & 1, a.status, 100000000ull);
    return;
  }
  if (tid < R) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, red_m[w * R + tid]);
    float Ls = 0.f;
    if (M != -INFINITY)
#pragma unroll
      for (int w = 0; w < 4; ++w) Ls += red_l[w * R + tid] * ex2(red_m[w * R + tid] - M);
    row_M[tid] = M;
    row_L[tid] = Ls;
  }
  consumer_sync<NCONS>();
  // every slab group writes its O, rescaled to the CTA max, into its own
  // [R][D] slice (the stage ring is free now); the slices are then summed in
  // a fixed order
  float* comb = reinterpret_cast<float*>(smem);
  {
    float fac[NQT][2];
    const float unlift = pow2i(-k_run);  // O carries 2^k_run (1 but for quantized V near the f16 limit)
#pragma unroll
    for (int j = 0; j < NQT; ++j)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float M = row_M[8 * j + 2 * c + u];
        fac[j][u] = M == -INFINITY ? 0.f : ex2(m_run[j][u] - M) * unlift;
      }
    float* mine = comb + pair * R * D;
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
      for (int j = 0; j < NQT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int qr = 8 * j + 2 * c + (e & 1), hi = e >> 1;
          int d;
          if constexpr (KV == KIND_BF16 || Cfg::V_SMEM) d = half * DH + 16 * mt + r + 8 * hi;
          else d = half * DH + 32 * (mt >> 1) + 4 * r + 2 * (mt & 1) + hi;
          mine[qr * D + d] = o[mt][j][e] * fac[j][e & 1];
        }
  }
  consumer_sync<NCONS>();
  const bool final_out = (nsplit == 1);
  const int64_t part0 = (static_cast<int64_t>(b) * a.H + h) * a.target;
  const int64_t part = part0 + split;
  for (int idx = tid; idx < R_real * (D / 4); idx += NCONS) {
    const int qr = idx / (D / 4), d = (idx % (D / 4)) * 4;
    float4 v = *reinterpret_cast<const float4*>(comb + qr * D + d);
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(comb + (w * R + qr) * D + d);
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    if (final_out) {
      const float L = row_L[qr];
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const int t = qr / a.G, g = qr % a.G;
      __nv_bfloat16* dst = a.out + ((static_cast<int64_t>(b) * a.T + t) * a.Hq + h * a.G + g) * D + d;
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(pack_bf16x2(v.x * inv, v.y * inv), pack_bf16x2(v.z * inv, v.w * inv));
    } else {
      *reinterpret_cast<float4*>(a.ws_acc + (part * R + qr) * D + d) = v;
    }
  }
  if (tid < R_real) {
    if (final_out) {
      if (a.lse) {
        const int t = tid / a.G, g = tid % a.G;
        const float L = row_L[tid];
        a.lse[(static_cast<int64_t>(b) * a.T + t) * a.Hq + h * a.G + g] =
            L > 0.f ? (row_M[tid] + log2f(L)) * kLn2 : -INFINITY;
      }
    } else {
      a.ws_ml[part * R + tid] = make_float2(row_M[tid], row_L[tid]);
    }
  }
}

// ---- log-sum-exp merge of the splits (separate launch) ----------------------------
// Split s of (row b, KV head h) holds (m_s, l_s, acc_s) for every query row;
// M = max_s m_s, L = sum_s l_s 2^(m_s - M), out = sum_s acc_s 2^(m_s - M) / L,
// lse = (M + log2 L) ln 2: the softmax over the union of the splits' keys.
// One CTA per (b, h, 32-dim slice), so a row's merge is spread over D / 32
// SMs; it recomputes the decode's split plan from the same frontiers and
// returns at once for rows the decode finished in one split.  Launched with
// programmatic stream serialization right behind the decode: everything
// before the wait overlaps the decode's tail.
template <int D, int NQT>
__global__ void __launch_bounds__(256) merge_kernel(DecodeArgs a) {
  constexpr int R = 8 * NQT;
  __shared__ int s_F[8];
  __shared__ float2 sml[R * kMaxSplits];
  __shared__ float sw[R * kMaxSplits];
  const int b = blockIdx.x, h = blockIdx.y, d0 = blockIdx.z * 32, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid < a.B) {
    const int F = a.frontiers[tid], row = a.table_rows[tid];
    const bool ok = F >= 0 && F <= a.L * 64 && row >= 0 && row < a.C && (a.k_new == nullptr || F >= a.T);
    s_F[tid] = ok ? F : 0;
  }
  __syncthreads();
  int total = 0, maxp = 0;
  for (int bb = 0; bb < a.B; ++bb) {
    const int np = (s_F[bb] + 63) >> 6;
    total += np;
    maxp = max(maxp, np);
  }
  const int chunk = a.nseg > 0 ? piece_chunk(s_F, a, total, maxp) : wave_chunk(s_F, a.B, total, maxp, a.target);
  const int nsplit = max(1, (((s_F[b] + 63) >> 6) + chunk - 1) / chunk);
  griddep_wait();
  griddep_launch_dependents();
  if (nsplit <= 1) return;  // the decode wrote this row's output
  const int R_real = a.T * a.G;
  const int64_t part0 = (static_cast<int64_t>(b) * a.H + h) * a.target;
  // item = (query row, 4 dims of the slice); four threads share an item and
  // take every fourth split, all of their loads in flight together.  The
  // accumulators of a thread's first item are loaded before the (m, l)
  // weights are known, so the two reads overlap.
  const int sub = tid & 3;
  const int64_t stride = static_cast<int64_t>(R) * D / 4;
  auto load_item = [&](int item, float4 (&v)[kMaxSplits / 4]) {
    const int qr = item >> 3, d = d0 + (item & 7) * 4;
    const float4* src = reinterpret_cast<const float4*>(a.ws_acc + (part0 * R + qr) * D + d);
#pragma unroll
    for (int u = 0; u < kMaxSplits / 4; ++u) {
      const int k = sub + 4 * u;
      v[u] = k < nsplit ? __ldcg(src + k * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  float4 v[kMaxSplits / 4];
  if ((tid >> 2) < R_real * 8) load_item(tid >> 2, v);
  for (int x = tid; x < R_real * nsplit; x += 256) {
    const int qr = x / nsplit, k = x - qr * nsplit;
    sml[x] = __ldcg(&a.ws_ml[(part0 + k) * R + qr]);
  }
  __syncthreads();
  for (int qr = warp; qr < R_real; qr += 8) {  // one warp per row, one lane per split
    const float2 ml = lane < nsplit ? sml[qr * nsplit + lane] : make_float2(-INFINITY, 0.f);
    float M = ml.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float e = M == -INFINITY ? 0.f : ex2(ml.x - M);
    float Ls = ml.y * e;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
    if (lane < nsplit) sw[qr * nsplit + lane] = Ls > 0.f ? e / Ls : 0.f;
    if (lane == 0 && a.lse && blockIdx.z == 0) {
      const int t = qr / a.G, g = qr % a.G;
      a.lse[(static_cast<int64_t>(b) * a.T + t) * a.Hq + h * a.G + g] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    }
  }
  __syncthreads();
  for (int item = tid >> 2; item < R_real * 8; item += 64) {
    if (item != (tid >> 2)) load_item(item, v);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int qr = item >> 3;
#pragma unroll
    for (int u = 0; u < kMaxSplits / 4; ++u) {
      const int k = sub + 4 * u;
      const float w = k < nsplit ? sw[qr * nsplit + k] : 0.f;
      acc.x = fmaf(w, v[u].x, acc.x);
      acc.y = fmaf(w, v[u].y, acc.y);
      acc.z = fmaf(w, v[u].z, acc.z);
      acc.w = fmaf(w, v[u].w, acc.w);
    }
    // the four shares (lanes 4k .. 4k + 3) in a fixed order: (0 + 1) + (2 + 3)
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    if (sub == 0) {
      const int d = d0 + (item & 7) * 4;
      const int t = qr / a.G, g = qr % a.G;
      __nv_bfloat16* dst = a.out + ((static_cast<int64_t>(b) * a.T + t) * a.Hq + h * a.G + g) * D + d;
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
  }
}

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
  cudaError_t e = launch_pdl(k, grid, dim3(Cfg::THREADS), Cfg::SMEM, s, tk, tv, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(merge_kernel<D, NQT>, dim3(a.B, a.H, D / 32), dim3(256), 0, s, a);
}

// Bytes of the stage ring, which the final combine and the merge reuse.
template <int KK, int KV, int D, int NQT>
int decode_ring_bytes() {
  using Cfg = DecodeCfg<KK, KV, D, NQT>;
  return Cfg::NSTAGE * Cfg::STAGE;
}

template <int KK, int KV, int D, int NQT>
int decode_ctas_per_sm() {
  using Cfg = DecodeCfg<KK, KV, D, NQT>;
  static int cached = 0;
  if (!cached) {
    auto k = decode_kernel<KK, KV, D, NQT>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, Cfg::THREADS, Cfg::SMEM) != cudaSuccess || n < 1)
      n = 1;
    cached = n;
  }
  return cached;
}

// Per-profile entry points (defined in decode_<profile>.cu).
using DecodeFn = cudaError_t (*)(const nk_pool*, int layer, const DecodeArgs&, int nqt, dim3 grid,
                                 cudaStream_t);
using OccFn = int (*)(int D, int nqt, int* ring_bytes);

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
int decode_occupancy(int D, int nqt, int* ring_bytes) {
#define NK_CASE(DD, Q)                                     \
  if (D == DD && nqt == Q) {                               \
    *ring_bytes = decode_ring_bytes<KK, KV, DD, Q>();      \
    return decode_ctas_per_sm<KK, KV, DD, Q>();            \
  }
  NK_CASE(64, 1) NK_CASE(64, 2) NK_CASE(64, 4)
  NK_CASE(128, 1) NK_CASE(128, 2) NK_CASE(128, 4)
  NK_CASE(256, 1) NK_CASE(256, 2)
#undef NK_CASE
  *ring_bytes = 0;
  return 1;
}

cudaError_t decode_bf16(const nk_pool*, int, const DecodeArgs&, int, dim3, cudaStream_t);
cudaError_t decode_int8(const nk_pool*, int, const DecodeArgs&, int, dim3, cudaStream_t);
cudaError_t decode_fp8(const nk_pool*, int, const DecodeArgs&, int, dim3, cudaStream_t);
cudaError_t decode_nvfp4(const nk_pool*, int, const DecodeArgs&, int, dim3, cudaStream_t);
cudaError_t decode_k8v4(const nk_pool*, int, const DecodeArgs&, int, dim3, cudaStream_t);
// The tcgen05 decode (vdecode.cu) for 17..32 query rows per KV head over
// pages whose codes are exact f16 operands (FP8-row, NVFP4-G16, K8V4); one
// CTA per SM.  nullptr for other profiles / shapes.
DecodeFn vdecode_for(int profile, int D, int nqt);
int occupancy_bf16(int, int, int*);
int occupancy_int8(int, int, int*);
int occupancy_fp8(int, int, int*);
int occupancy_nvfp4(int, int, int*);
int occupancy_k8v4(int, int, int*);

}  // namespace nk
