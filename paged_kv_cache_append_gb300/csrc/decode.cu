// decode.cu -- host side of the paged decode attention: split plan,
// workspace layout and launch.
//
// Workspace: [per-split (m, l) of every query row] [per-split unnormalised
// accumulators].  Every slot the merge reads is written first by the same
// call, so the workspace needs no initialisation.
#include <cmath>

#include "decode.cuh"

namespace nk {

struct DecodePlan {
  int nqt, R, target, ring_bytes;
  int ctas = 0;  // CTAs per KV head (grid x)
  int nseg = 0;  // > 0: pieces per head, several per CTA
  size_t ws_ml_bytes, ws_bytes;
  DecodeFn fn;
};

static void plan_sizes(DecodePlan* pl, int B, int H, int D) {
  const size_t parts = static_cast<size_t>(B) * H * pl->target * pl->R;
  pl->ws_ml_bytes = (parts * sizeof(float2) + 255) / 256 * 256;
  pl->ws_bytes = pl->ws_ml_bytes + parts * D * sizeof(float);
}

static int make_plan(const nk_pool* p, int B, int T, int Hq, DecodePlan* pl) {
  const int H = p->desc.num_kv_heads, D = p->desc.head_dim;
  if (Hq < 1 || Hq % H) return fail(NK_ERR_SHAPE, "Hq must be a positive multiple of num_kv_heads");
  if (B < 1 || B > p->desc.max_concurrency) return fail(NK_ERR_SHAPE, "B must be in [1, C]");
  if (T < 1) return fail(NK_ERR_SHAPE, "T must be >= 1");
  const int Rr = T * (Hq / H);
  pl->nqt = Rr <= 8 ? 1 : Rr <= 16 ? 2 : Rr <= 32 ? 4 : 0;
  if (!pl->nqt) return fail(NK_ERR_UNSUPPORTED, "T * Hq / num_kv_heads must be <= 32");
  const DecodeFn vfn = vdecode_for(p->desc.profile, D, pl->nqt);
  if (D == 256 && pl->nqt == 4 && !vfn)
    return fail(NK_ERR_UNSUPPORTED,
                "head_dim 256 with T * Hq / num_kv_heads > 16 needs the FP8-row, NVFP4-G16 or K8V4 profile");
  pl->R = 8 * pl->nqt;
  OccFn occ;
  switch (p->desc.profile) {
    case NK_BF16: pl->fn = decode_bf16; occ = occupancy_bf16; break;
    case NK_INT8_G64: pl->fn = decode_int8; occ = occupancy_int8; break;
    case NK_FP8_E4M3_ROW: pl->fn = decode_fp8; occ = occupancy_fp8; break;
    case NK_NVFP4_G16: pl->fn = decode_nvfp4; occ = occupancy_nvfp4; break;
    default: pl->fn = decode_k8v4; occ = occupancy_k8v4; break;
  }
  int per_sm = occ(D, pl->nqt, &pl->ring_bytes);
  if (vfn) {  // 17..32 query rows over exact-f16 codes: the tcgen05 kernel, one CTA per SM
    pl->fn = vfn;
    per_sm = 1;
  }
  pl->target = p->num_sms * per_sm / H;
  if (pl->target < 1) pl->target = 1;
  // A budget below B (many KV heads) leaves every row one split, which still
  // needs one CTA per row: the grid never has fewer CTAs than rows.
  pl->ctas = pl->target > B ? pl->target : B;
  if (vfn && D <= 128) {
    // the transposed tcgen05 kernel takes several (row, page range) pieces
    // per CTA, so that equal rows still fill every SM; a row has at most
    // kMaxSplits pieces, each with its own partial slot
    pl->nseg = 4 * pl->ctas;
    pl->target = pl->nseg < kMaxSplits ? pl->nseg : kMaxSplits;
  }
  plan_sizes(pl, B, H, D);
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

namespace nk {

// Shared by the decode entry points: checks, plan, arguments, launch.
// k_new / v_new non-null: fused append of the T new tokens first.
static int run_decode(const void* q, int32_t Hq, const nk_pool* pool, int32_t layer,
                      const int32_t* block_tables, const int32_t* table_rows,
                      const int32_t* frontiers, const void* k_new, const void* v_new, int32_t B,
                      int32_t T, float softmax_scale, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, cudaStream_t s, const char* what) {
  if (!q || !pool || !block_tables || !table_rows || !frontiers || !out)
    return fail(NK_ERR_INVALID_ARG, std::string("null argument to ") + what);
  if (!std::isfinite(softmax_scale)) return fail(NK_ERR_INVALID_ARG, "softmax_scale is not finite");
  if (layer < 0 || layer >= pool->desc.num_layers) return fail(NK_ERR_SHAPE, "layer out of range");
  if (!aligned16(q) || !aligned16(out)) return fail(NK_ERR_ALIGN, "q / out must be 16-byte aligned");
  if ((k_new != nullptr) != (v_new != nullptr)) return fail(NK_ERR_INVALID_ARG, "k and v come together");
  if (k_new && (!aligned16(k_new) || !aligned16(v_new)))
    return fail(NK_ERR_ALIGN, "k / v must be 16-byte aligned");
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
  a.ws_ml = reinterpret_cast<float2*>(workspace);
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
  a.nseg = pl.nseg;
  a.ctas = pl.ctas;
  a.head_major = pool->desc.order == NK_HEAD_MAJOR;
  if (k_new) {
    a.k_new = static_cast<const __nv_bfloat16*>(k_new);
    a.v_new = static_cast<const __nv_bfloat16*>(v_new);
    a.kc_w = static_cast<uint8_t*>(pool->ptrs[layer * np + 0]);
    a.vc_w = static_cast<uint8_t*>(pool->ptrs[layer * np + 1]);
    a.ks_w = np == 4 ? static_cast<uint8_t*>(pool->ptrs[layer * np + 2]) : nullptr;
    a.vs_w = np == 4 ? static_cast<uint8_t*>(pool->ptrs[layer * np + 3]) : nullptr;
  }
  cudaError_t e = pl.fn(pool, layer, a, pl.nqt, dim3(pl.ctas, a.H), s);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return NK_OK;
}

}  // namespace nk

extern "C" int nk_paged_decode_attention(const void* q, int32_t Hq, const nk_pool* pool,
                                         int32_t layer, const int32_t* block_tables,
                                         const int32_t* table_rows, const int32_t* frontiers,
                                         int32_t B, int32_t T, float softmax_scale, void* out,
                                         float* lse, void* workspace, size_t workspace_bytes,
                                         void* stream) {
  clear_error();
  return run_decode(q, Hq, pool, layer, block_tables, table_rows, frontiers, nullptr, nullptr, B, T,
                    softmax_scale, out, lse, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream), "nk_paged_decode_attention");
}

extern "C" int nk_paged_append_decode_attention(const void* q, int32_t Hq, nk_pool* pool,
                                                int32_t layer, const int32_t* block_tables,
                                                const int32_t* table_rows,
                                                const int32_t* frontiers, const void* k,
                                                const void* v, int32_t B, int32_t T,
                                                float softmax_scale, void* out, float* lse,
                                                void* workspace, size_t workspace_bytes,
                                                void* stream) {
  clear_error();
  if (!k || !v) return fail(NK_ERR_INVALID_ARG, "null k / v to nk_paged_append_decode_attention");
  return run_decode(q, Hq, pool, layer, block_tables, table_rows, frontiers, k, v, B, T, softmax_scale,
                    out, lse, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                    "nk_paged_append_decode_attention");
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
    const size_t fixed = 512;  // alignment of the (m, l) block
    const size_t fit = max_ws > fixed ? (max_ws - fixed) / per_split : 0;
    if (fit < 1)
      return fail(NK_ERR_WORKSPACE, "one split of this call needs " + std::to_string(per_split + fixed) +
                                        " bytes of scratch; the static scratch holds " +
                                        std::to_string(max_ws));
    // Fewer partial slots per (row, KV head).  The slot count bounds the
    // splits of the plan (a budget below B gives every row one split, which
    // writes its output directly); the CTA count must still cover the splits,
    // so it never drops below B.
    pl.target = static_cast<int>(fit < static_cast<size_t>(pl.target) ? fit : pl.target);
    if (pl.nseg > 0) {
      if (pl.nseg > pl.target) pl.nseg = pl.target;  // every row's pieces still fit its slots
    } else {
      pl.ctas = pl.target > B ? pl.target : B;
    }
    plan_sizes(&pl, B, H, D);
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
  a.ws_ml = reinterpret_cast<float2*>(scratch);
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
  a.nseg = pl.nseg;
  a.ctas = pl.ctas;
  a.head_major = pool->desc.order == NK_HEAD_MAJOR;
  cudaError_t e = pl.fn(pool, layer, a, pl.nqt, dim3(pl.ctas, a.H), s);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return NK_OK;
}

}  // namespace nk
