// decode.cu -- host side of the paged decode attention and the log-sum-exp
// merge of split-K partials.
//
// Merge (split-K over pages): with per-split running max m_s (base 2), sum
// l_s and unnormalised accumulator acc_s,
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),
//   out = sum_s acc_s 2^(m_s - M) / L,  lse = (M + log2 L) ln 2,
// which is exactly the softmax over the union of the splits' keys.
#include <cmath>

#include "decode.cuh"

namespace nk {

// One CTA per (64 head dims, KV head, row).  Warps first turn each query's
// split statistics into weights w_s = 2^(m_s - M) / L (shared memory), then
// every thread sums weighted partials for a few (query, dim) outputs with
// coalesced loads over the dims.
constexpr int kMergeDims = 64;

__global__ void __launch_bounds__(128) merge_kernel(DecodeArgs a, int R, int D) {
  extern __shared__ float w_s[];  // [T*G][target]
  __shared__ int s_F[8];
  const int b = blockIdx.z, h = blockIdx.y, d0 = blockIdx.x * kMergeDims;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < a.B) {
    const int F = a.frontiers[tid], row = a.table_rows[tid];
    s_F[tid] = (F >= 0 && F <= a.L * 64 && row >= 0 && row < a.C) ? F : 0;
  }
  __syncthreads();
  int total = 0;
  for (int bb = 0; bb < a.B; ++bb) total += (s_F[bb] + 63) >> 6;
  const int chunk = split_chunk(total, a.target, a.B);
  const int ns = (((s_F[b] + 63) >> 6) + chunk - 1) / chunk;
  if (ns == 1) return;  // the decode CTA of this row wrote out / lse itself
  const int Rr = a.T * a.G;
  const int64_t part0 = (static_cast<int64_t>(b) * a.H + h) * a.target;
  for (int qr = warp; qr < Rr; qr += 4) {
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, a.ws_ml[(part0 + s) * R + qr].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    if (M != -INFINITY)
      for (int s = lane; s < ns; s += 32) {
        const float2 ml = a.ws_ml[(part0 + s) * R + qr];
        L += ml.y * ex2(ml.x - M);
      }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int s = lane; s < ns; s += 32)
      w_s[qr * a.target + s] = L > 0.f ? ex2(a.ws_ml[(part0 + s) * R + qr].x - M) * inv : 0.f;
    if (lane == 0 && blockIdx.x == 0 && a.lse) {
      const int t = qr / a.G, g = qr % a.G;
      a.lse[(static_cast<int64_t>(b) * a.T + t) * a.Hq + h * a.G + g] =
          L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
  }
  __syncthreads();
  const int nd = min(kMergeDims, D - d0);
  for (int i = tid; i < Rr * nd; i += 128) {
    const int qr = i / nd, d = d0 + i % nd;
    const float* src = a.ws_acc + (part0 * R + qr) * D + d;
    const float* w = w_s + qr * a.target;
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    int s = 0;
    for (; s + 4 <= ns; s += 4) {
      acc0 = fmaf(w[s], src[static_cast<int64_t>(s) * R * D], acc0);
      acc1 = fmaf(w[s + 1], src[static_cast<int64_t>(s + 1) * R * D], acc1);
      acc2 = fmaf(w[s + 2], src[static_cast<int64_t>(s + 2) * R * D], acc2);
      acc3 = fmaf(w[s + 3], src[static_cast<int64_t>(s + 3) * R * D], acc3);
    }
    for (; s < ns; ++s) acc0 = fmaf(w[s], src[static_cast<int64_t>(s) * R * D], acc0);
    const int t = qr / a.G, g = qr % a.G;
    a.out[((static_cast<int64_t>(b) * a.T + t) * a.Hq + h * a.G + g) * D + d] =
        __float2bfloat16_rn((acc0 + acc1) + (acc2 + acc3));
  }
}

// Launches the merge; its dynamic shared memory holds T*G x target weights.
static cudaError_t launch_merge(const DecodeArgs& a, int R, int D, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(a.T) * a.G * a.target * sizeof(float);
  static size_t attr = 0;
  if (smem > 48 * 1024 && smem > attr) {
    cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr = smem;
  }
  merge_kernel<<<dim3((D + kMergeDims - 1) / kMergeDims, a.H, a.B), 128, smem, s>>>(a, R, D);
  return cudaGetLastError();
}

struct DecodePlan {
  int nqt, R, target;
  size_t ws_ml_bytes, ws_bytes;
  DecodeFn fn;
};

static int make_plan(const nk_pool* p, int B, int T, int Hq, DecodePlan* pl) {
  const int H = p->desc.num_kv_heads, D = p->desc.head_dim;
  if (Hq < 1 || Hq % H) return fail(NK_ERR_SHAPE, "Hq must be a positive multiple of num_kv_heads");
  if (B < 1 || B > p->desc.max_concurrency) return fail(NK_ERR_SHAPE, "B must be in [1, C]");
  if (T < 1) return fail(NK_ERR_SHAPE, "T must be >= 1");
  const int Rr = T * (Hq / H);
  pl->nqt = Rr <= 8 ? 1 : Rr <= 16 ? 2 : Rr <= 32 ? 4 : 0;
  if (!pl->nqt) return fail(NK_ERR_UNSUPPORTED, "T * Hq / num_kv_heads must be <= 32");
  if (D == 256 && pl->nqt == 4)
    return fail(NK_ERR_UNSUPPORTED, "head_dim 256 supports T * Hq / num_kv_heads <= 16");
  pl->R = 8 * pl->nqt;
  OccFn occ;
  switch (p->desc.profile) {
    case NK_BF16: pl->fn = decode_bf16; occ = occupancy_bf16; break;
    case NK_INT8_G64: pl->fn = decode_int8; occ = occupancy_int8; break;
    case NK_FP8_E4M3_ROW: pl->fn = decode_fp8; occ = occupancy_fp8; break;
    case NK_NVFP4_G16: pl->fn = decode_nvfp4; occ = occupancy_nvfp4; break;
    default: pl->fn = decode_k8v4; occ = occupancy_k8v4; break;
  }
  const int per_sm = occ(D, pl->nqt);
  pl->target = p->num_sms * per_sm / H;
  if (pl->target < 1) pl->target = 1;
  const size_t parts = static_cast<size_t>(B) * H * pl->target * pl->R;
  pl->ws_ml_bytes = (parts * sizeof(float2) + 255) / 256 * 256;
  pl->ws_bytes = pl->ws_ml_bytes + parts * D * sizeof(float);
  return NK_OK;
}

}  // namespace nk

using namespace nk;

extern "C" int nk_decode_workspace_bytes(const nk_pool* pool, int32_t B, int32_t T, int32_t Hq,
                                         size_t* bytes) {
  clear_error();
  if (!pool || !bytes) return fail(NK_ERR_INVALID_ARG, "null argument");
  DecodePlan pl;
  int rc = make_plan(pool, B, T, Hq, &pl);
  if (rc) return rc;
  *bytes = pl.ws_bytes;
  return NK_OK;
}

extern "C" int nk_paged_decode_attention(const void* q, int32_t Hq, const nk_pool* pool,
                                         int32_t layer, const int32_t* block_tables,
                                         const int32_t* table_rows, const int32_t* frontiers,
                                         int32_t B, int32_t T, float softmax_scale, void* out,
                                         float* lse, void* workspace, size_t workspace_bytes,
                                         void* stream) {
  clear_error();
  if (!q || !pool || !block_tables || !table_rows || !frontiers || !out)
    return fail(NK_ERR_INVALID_ARG, "null argument to nk_paged_decode_attention");
  if (!std::isfinite(softmax_scale)) return fail(NK_ERR_INVALID_ARG, "softmax_scale is not finite");
  if (layer < 0 || layer >= pool->desc.num_layers) return fail(NK_ERR_SHAPE, "layer out of range");
  if (!aligned16(q) || !aligned16(out)) return fail(NK_ERR_ALIGN, "q / out must be 16-byte aligned");
  DecodePlan pl;
  int rc = make_plan(pool, B, T, Hq, &pl);
  if (rc) return rc;
  if (!workspace || workspace_bytes < pl.ws_bytes)
    return fail(NK_ERR_WORKSPACE, "workspace needs " + std::to_string(pl.ws_bytes) + " bytes");
  if (!aligned16(workspace)) return fail(NK_ERR_ALIGN, "workspace must be 16-byte aligned");
  DecodeArgs a;
  const int np = pool->n_planes;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.tables = block_tables;
  a.table_rows = table_rows;
  a.frontiers = frontiers;
  a.ks = np == 4 ? static_cast<const uint8_t*>(pool->ptrs[layer * np + 2]) : nullptr;
  a.vs = np == 4 ? static_cast<const uint8_t*>(pool->ptrs[layer * np + 3]) : nullptr;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.ws_ml = static_cast<float2*>(workspace);
  a.ws_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + pl.ws_ml_bytes);
  a.status = pool->status;
  a.softmax_scale = softmax_scale;
  a.B = B;
  a.T = T;
  a.Hq = Hq;
  a.H = pool->desc.num_kv_heads;
  a.G = Hq / a.H;
  a.L = pool->L;
  a.M = pool->M;
  a.C = pool->desc.max_concurrency;
  a.target = pl.target;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = pl.fn(pool, layer, a, pl.nqt, dim3(pl.target, a.H), s);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  e = launch_merge(a, pl.R, pool->desc.head_dim, s);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return NK_OK;
}

namespace nk {

// Decode + merge whose split-K partials live in a caller-given scratch area
// of at most `max_ws` bytes: the split target is lowered until the partials
// fit.  Used by the entry point that allocates nothing (decode_noalloc.cu).
int decode_with_scratch(const void* q, int32_t Hq, const nk_pool* pool, int32_t layer,
                        const int32_t* block_tables, const int32_t* table_rows,
                        const int32_t* frontiers, int32_t B, int32_t T, float softmax_scale,
                        void* out, float* lse, void* scratch, size_t max_ws, cudaStream_t s) {
  if (!q || !pool || !block_tables || !table_rows || !frontiers || !out || !scratch)
    return fail(NK_ERR_INVALID_ARG, "null argument to the static-scratch decode");
  if (!std::isfinite(softmax_scale)) return fail(NK_ERR_INVALID_ARG, "softmax_scale is not finite");
  if (layer < 0 || layer >= pool->desc.num_layers) return fail(NK_ERR_SHAPE, "layer out of range");
  if (!aligned16(q) || !aligned16(out)) return fail(NK_ERR_ALIGN, "q / out must be 16-byte aligned");
  DecodePlan pl;
  int rc = make_plan(pool, B, T, Hq, &pl);
  if (rc) return rc;
  const int H = pool->desc.num_kv_heads, D = pool->desc.head_dim;
  const size_t per_split = static_cast<size_t>(B) * H * pl.R * (sizeof(float2) + D * sizeof(float));
  if (pl.ws_bytes > max_ws) {
    const size_t fit = (max_ws - 256) / per_split;
    if (fit < 1)
      return fail(NK_ERR_WORKSPACE, "one split of this call needs " + std::to_string(per_split + 256) +
                                        " bytes of scratch; the static scratch holds " +
                                        std::to_string(max_ws));
    pl.target = static_cast<int>(fit < static_cast<size_t>(pl.target) ? fit : pl.target);
    const size_t parts = static_cast<size_t>(B) * H * pl.target * pl.R;
    pl.ws_ml_bytes = (parts * sizeof(float2) + 255) / 256 * 256;
    pl.ws_bytes = pl.ws_ml_bytes + parts * D * sizeof(float);
  }
  DecodeArgs a;
  const int np = pool->n_planes;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.tables = block_tables;
  a.table_rows = table_rows;
  a.frontiers = frontiers;
  a.ks = np == 4 ? static_cast<const uint8_t*>(pool->ptrs[layer * np + 2]) : nullptr;
  a.vs = np == 4 ? static_cast<const uint8_t*>(pool->ptrs[layer * np + 3]) : nullptr;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.ws_ml = static_cast<float2*>(scratch);
  a.ws_acc = reinterpret_cast<float*>(static_cast<char*>(scratch) + pl.ws_ml_bytes);
  a.status = pool->status;
  a.softmax_scale = softmax_scale;
  a.B = B;
  a.T = T;
  a.Hq = Hq;
  a.H = H;
  a.G = Hq / H;
  a.L = pool->L;
  a.M = pool->M;
  a.C = pool->desc.max_concurrency;
  a.target = pl.target;
  cudaError_t e = pl.fn(pool, layer, a, pl.nqt, dim3(pl.target, a.H), s);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  e = launch_merge(a, pl.R, D, s);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return NK_OK;
}

}  // namespace nk
