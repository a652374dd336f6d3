// append.cu -- growing-cache KV append with fused quantization.
//
// "Paged KV cache" maintainer design page: a token at logical position pos of
// a table row lives in page group g = block_table[pos >> 6] at page offset
// o = pos & 63 (consumer view section, translation), and its codes and scales
// share that g in every plane (page grouping section).  The page names the
// persistent codec "kv_cache_append" but leaves its rules open; the rules
// implemented here are this library's (see nk.h, nk_profile):
//   INT8-G64  s = fp16(fp32(amax/127)), q = clamp(RNE(x/s), -127, 127)
//   FP8-row   s = fp16(fp32(amax/448)), c = E4M3FN RNE satfinite (x/s)
//   NVFP4-G16 s8 = E4M3FN RNE satfinite (fp32(amax/6)), c = E2M1 RNE satfinite (x/s8)
// fp32 quotients (__fdiv_rn) followed by one RNE conversion give the exactly
// rounded quotient for these operand widths, so codes are bit-exact.
//
// One warp encodes one (row b, token t, KV head h): both K and V (encode.cuh).
#include "encode.cuh"

namespace nk {

struct AppendArgs {
  const int32_t* tables;
  const int32_t* table_rows;
  const int32_t* write_pos;
  const int32_t* counts;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  uint8_t* kc;  // K code plane
  uint8_t* vc;  // V code plane
  uint8_t* ks;  // K scale plane (nullptr for BF16)
  uint8_t* vs;  // V scale plane
  int* status;
  int B, T, H, L, M, C;
  int head_major;  // plane order
};

template <int KK, int KV, int D>
__global__ void __launch_bounds__(128) append_kernel(AppendArgs a) {
  griddep_wait();  // launched with programmatic stream serialization
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (gw >= a.B * a.T * a.H) return;
  const int h = gw % a.H;
  const int t = (gw / a.H) % a.T;
  const int b = gw / (a.H * a.T);
  const int n = a.counts ? a.counts[b] : a.T;
  if (t >= n) return;
  const int row = a.table_rows[b];
  const int pos = a.write_pos[b] + t;
  // Out-of-range rows, positions and page ids are skipped, never written.
  if (row < 0 || row >= a.C || pos < 0 || pos >= a.L * 64) {
    if (lane == 0) set_status(a.status, NK_STATUS_FRONTIER);
    return;
  }
  const int g = a.tables[static_cast<int64_t>(row) * a.L + (pos >> 6)];
  if (g < 0 || g >= a.M) {
    if (lane == 0) set_status(a.status, NK_STATUS_PAGE_RANGE);
    return;
  }
  const int64_t token_row = tile_row(g, h, a.H, a.M, a.head_major) + (pos & 63);
  const int64_t src = ((static_cast<int64_t>(b) * a.T + t) * a.H + h) * D;

  constexpr int KCB = code_row_bytes<KK>(D), VCB = code_row_bytes<KV>(D);
  constexpr int KSB = scale_row_bytes<KK>(D), VSB = scale_row_bytes<KV>(D);
  encode_row<KK, D>(a.k + src, a.kc + token_row * KCB, a.ks ? a.ks + token_row * KSB : nullptr, lane);
  encode_row<KV, D>(a.v + src, a.vc + token_row * VCB, a.vs ? a.vs + token_row * VSB : nullptr, lane);
}

template <int KK, int KV>
static void launch_d(int D, const AppendArgs& a, cudaStream_t s) {
  const int warps = a.B * a.T * a.H;
  const dim3 grid((warps + 3) / 4), block(128);
  if (D == 64) launch_pdl(append_kernel<KK, KV, 64>, grid, block, 0, s, a);
  else if (D == 128) launch_pdl(append_kernel<KK, KV, 128>, grid, block, 0, s, a);
  else launch_pdl(append_kernel<KK, KV, 256>, grid, block, 0, s, a);
}

}  // namespace nk

using namespace nk;

extern "C" int nk_paged_kv_append(nk_pool* pool, int32_t layer, const int32_t* block_tables,
                                  const int32_t* table_rows, const int32_t* write_pos,
                                  const int32_t* counts, const void* k, const void* v, int32_t B,
                                  int32_t T, void* stream) {
  clear_error();
  if (!pool || !block_tables || !table_rows || !write_pos || !k || !v)
    return fail(NK_ERR_INVALID_ARG, "null argument to nk_paged_kv_append");
  if (layer < 0 || layer >= pool->desc.num_layers) return fail(NK_ERR_SHAPE, "layer out of range");
  if (B < 1 || B > pool->desc.max_concurrency) return fail(NK_ERR_SHAPE, "B must be in [1, C]");
  if (T < 1) return fail(NK_ERR_SHAPE, "T must be >= 1");
  if (!aligned16(k) || !aligned16(v)) return fail(NK_ERR_ALIGN, "k / v must be 16-byte aligned");
  if (static_cast<int64_t>(B) * T * pool->desc.num_kv_heads > (int64_t(1) << 30))
    return fail(NK_ERR_SHAPE, "too many token rows in one append");
  AppendArgs a;
  const int np = pool->n_planes;
  a.tables = block_tables;
  a.table_rows = table_rows;
  a.write_pos = write_pos;
  a.counts = counts;
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.kc = static_cast<uint8_t*>(pool->ptrs[layer * np + 0]);
  a.vc = static_cast<uint8_t*>(pool->ptrs[layer * np + 1]);
  a.ks = np == 4 ? static_cast<uint8_t*>(pool->ptrs[layer * np + 2]) : nullptr;
  a.vs = np == 4 ? static_cast<uint8_t*>(pool->ptrs[layer * np + 3]) : nullptr;
  a.status = pool->status;
  a.B = B;
  a.T = T;
  a.H = pool->desc.num_kv_heads;
  a.L = pool->L;
  a.M = pool->M;
  a.C = pool->desc.max_concurrency;
  a.head_major = pool->desc.order == NK_HEAD_MAJOR;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = pool->desc.head_dim;
  switch (pool->desc.profile) {
    case NK_BF16: launch_d<KIND_BF16, KIND_BF16>(D, a, s); break;
    case NK_INT8_G64: launch_d<KIND_INT8, KIND_INT8>(D, a, s); break;
    case NK_FP8_E4M3_ROW: launch_d<KIND_FP8, KIND_FP8>(D, a, s); break;
    case NK_NVFP4_G16: launch_d<KIND_NVFP4, KIND_NVFP4>(D, a, s); break;
    default: launch_d<KIND_FP8, KIND_NVFP4>(D, a, s); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return NK_OK;
}
