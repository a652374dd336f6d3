// pool.cu -- pool geometry, validation, TMA descriptors, status word, error
// text and the partial-tail copy-on-write of libnk.
//
// Geometry follows the "Paged KV cache" maintainer design page: P = 64,
// L = ceil(S/P), M in [max(L, C), C*L] (capacity section); page-major planes
// [X, P, H, N] with code plane X = D, INT8-G64 scale X = D/64, FP8-row scale
// X = 1, NVFP4 packed codes X = D/2 and scales X = D/16 (physical layout
// section).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "internal.h"

namespace nk {

static thread_local std::string t_error;

int fail(int code, const std::string& msg) {
  t_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  t_error = std::string(what) + ": " + cudaGetErrorString(e);
  return NK_ERR_CUDA;
}

void clear_error() { t_error.clear(); }

int profile_kinds(int profile, Kind* k, Kind* v) {
  switch (profile) {
    case NK_BF16: *k = *v = KIND_BF16; return NK_OK;
    case NK_INT8_G64: *k = *v = KIND_INT8; return NK_OK;
    case NK_FP8_E4M3_ROW: *k = *v = KIND_FP8; return NK_OK;
    case NK_NVFP4_G16: *k = *v = KIND_NVFP4; return NK_OK;
    case NK_K8V4: *k = KIND_FP8; *v = KIND_NVFP4; return NK_OK;
    default: return fail(NK_ERR_INVALID_ARG, "unknown KV profile " + std::to_string(profile));
  }
}

static PlaneGeom code_geom(Kind k, int D) {
  switch (k) {
    case KIND_BF16: return {2, D, 2 * D};
    case KIND_INT8:
    case KIND_FP8: return {1, D, D};
    default: return {1, D / 2, D / 2};
  }
}

static PlaneGeom scale_geom(Kind k, int D) {
  switch (k) {
    case KIND_INT8: return {2, D / 64, 2 * (D / 64)};
    case KIND_FP8: return {2, 1, 2};
    default: return {1, D / 16, D / 16};
  }
}

int plane_geoms(int profile, int D, int* n_planes, PlaneGeom g[4]) {
  Kind k, v;
  int rc = profile_kinds(profile, &k, &v);
  if (rc) return rc;
  if (D != 64 && D != 128 && D != 256)
    return fail(NK_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256, got " + std::to_string(D));
  g[0] = code_geom(k, D);
  g[1] = code_geom(v, D);
  if (k == KIND_BF16) {
    *n_planes = 2;
    g[2] = g[3] = {0, 0, 0};
  } else {
    *n_planes = 4;
    g[2] = scale_geom(k, D);
    g[3] = scale_geom(v, D);
  }
  return NK_OK;
}

int device_sm_count(int device) {
  static std::mutex mu;
  static int cache[64] = {0};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return 0;
  if (!cache[device]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    cache[device] = n;
  }
  return cache[device];
}

// One status word per device.  Its host-side name is only a stand-in, so the
// kernels get its device address from cudaGetSymbolAddress.
static __device__ int g_status_word;

int* status_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

static int check_desc(const nk_pool_desc* d) {
  if (!d) return fail(NK_ERR_INVALID_ARG, "desc is NULL");
  if (d->num_layers < 1 || d->num_kv_heads < 1 || d->max_context < 1)
    return fail(NK_ERR_SHAPE, "num_layers, num_kv_heads and max_context must be >= 1");
  if (d->max_concurrency < 1 || d->max_concurrency > 8)
    return fail(NK_ERR_SHAPE, "max_concurrency must be in 1..8");
  if (d->order != NK_PAGE_MAJOR && d->order != NK_HEAD_MAJOR)
    return fail(NK_ERR_INVALID_ARG, "order must be NK_PAGE_MAJOR or NK_HEAD_MAJOR");
  if (d->flags & ~NK_POOL_CHECK_BOUNDS) return fail(NK_ERR_INVALID_ARG, "unknown pool flags");
  return NK_OK;
}

}  // namespace nk

using namespace nk;

extern "C" int nk_version(void) { return 100; }

extern "C" const char* nk_last_error(void) { return t_error.c_str(); }

extern "C" int nk_pool_capacity_bounds(const nk_pool_desc* desc, int32_t* m_min, int32_t* m_max) {
  clear_error();
  int rc = check_desc(desc);
  if (rc) return rc;
  if (!m_min || !m_max) return fail(NK_ERR_INVALID_ARG, "output pointers are NULL");
  const int64_t L = (static_cast<int64_t>(desc->max_context) + NK_PAGE_TOKENS - 1) / NK_PAGE_TOKENS;
  const int64_t C = desc->max_concurrency;
  *m_min = static_cast<int32_t>(L > C ? L : C);
  *m_max = static_cast<int32_t>(C * L);
  return NK_OK;
}

extern "C" int nk_pool_mtp_pages(int32_t M, int32_t C, int32_t draft_window, int32_t* pages) {
  clear_error();
  if (!pages) return fail(NK_ERR_INVALID_ARG, "output pointer is NULL");
  if (M < 1 || C < 1 || draft_window < 1) return fail(NK_ERR_RANGE, "M, C and the draft window must be >= 1");
  const int64_t lead = (static_cast<int64_t>(draft_window) - 1 + NK_PAGE_TOKENS - 1) / NK_PAGE_TOKENS;
  const int64_t n = static_cast<int64_t>(M) + static_cast<int64_t>(C) * lead;
  if (n > INT32_MAX) return fail(NK_ERR_RANGE, "page count does not fit int32");
  *pages = static_cast<int32_t>(n);
  return NK_OK;
}

extern "C" int nk_pages_needed(int32_t committed_frontier, int32_t provisional_frontier, int32_t* pages) {
  clear_error();
  if (!pages) return fail(NK_ERR_INVALID_ARG, "output pointer is NULL");
  if (committed_frontier < 0 || provisional_frontier < 0) return fail(NK_ERR_RANGE, "frontiers must be >= 0");
  const int64_t f = committed_frontier > provisional_frontier ? committed_frontier : provisional_frontier;
  *pages = static_cast<int32_t>((f + NK_PAGE_TOKENS - 1) / NK_PAGE_TOKENS);
  return NK_OK;
}

extern "C" int nk_pool_plane_bytes(const nk_pool_desc* desc, int32_t M, int32_t* n_planes,
                                   size_t bytes[4], size_t row_bytes[4]) {
  clear_error();
  int rc = check_desc(desc);
  if (rc) return rc;
  if (!n_planes || !bytes) return fail(NK_ERR_INVALID_ARG, "output pointers are NULL");
  if (M < 1) return fail(NK_ERR_RANGE, "M must be >= 1");
  PlaneGeom g[4];
  rc = plane_geoms(desc->profile, desc->head_dim, n_planes, g);
  if (rc) return rc;
  for (int i = 0; i < 4; ++i) {
    bytes[i] = i < *n_planes ? static_cast<size_t>(g[i].row_bytes) * NK_PAGE_TOKENS *
                                   desc->num_kv_heads * static_cast<size_t>(M)
                             : 0;
    if (row_bytes) row_bytes[i] = i < *n_planes ? g[i].row_bytes : 0;
  }
  return NK_OK;
}

// TMA descriptor of one code plane: a 2-D uint8 tensor of rows of row_bytes
// bytes (one row per (g, h, o) token), boxes of 64 rows x min(row_bytes, 128)
// bytes, swizzled so that rows of a box land in distinct shared-memory banks.
namespace nk {
int encode_code_tmap(CUtensorMap* m, void* base, int row_bytes, int64_t rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
      return fail(NK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  const int box_x = row_bytes < 128 ? row_bytes : 128;
  CUtensorMapSwizzle sw = box_x == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : box_x == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                        : CU_TENSOR_MAP_SWIZZLE_32B;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_x), 64u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(NK_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return NK_OK;
}
}  // namespace nk

extern "C" int nk_pool_create(const nk_pool_desc* desc, int32_t M, void* const* planes,
                              nk_pool** out) {
  clear_error();
  int rc = check_desc(desc);
  if (rc) return rc;
  if (!planes || !out) return fail(NK_ERR_INVALID_ARG, "planes / out is NULL");
  int32_t lo, hi;
  nk_pool_capacity_bounds(desc, &lo, &hi);
  if (M < lo || M > hi)
    return fail(NK_ERR_RANGE, "page groups M=" + std::to_string(M) + " outside [M_min=" +
                                  std::to_string(lo) + ", M_max=" + std::to_string(hi) + "]");
  int n_planes;
  PlaneGeom g[4];
  rc = plane_geoms(desc->profile, desc->head_dim, &n_planes, g);
  if (rc) return rc;
  const int64_t rows = static_cast<int64_t>(M) * desc->num_kv_heads * NK_PAGE_TOKENS;
  if (rows >= (int64_t(1) << 31)) return fail(NK_ERR_RANGE, "pool too large for 32-bit row index");
  for (int i = 0; i < desc->num_layers * n_planes; ++i) {
    if (!planes[i]) return fail(NK_ERR_INVALID_ARG, "plane pointer " + std::to_string(i) + " is NULL");
    if (!aligned16(planes[i]))
      return fail(NK_ERR_ALIGN, "plane pointer " + std::to_string(i) + " is not 16-byte aligned");
  }
  nk_pool* p = new (std::nothrow) nk_pool();
  if (!p) return fail(NK_ERR_INVALID_ARG, "out of host memory");
  p->desc = *desc;
  p->M = M;
  p->L = (desc->max_context + NK_PAGE_TOKENS - 1) / NK_PAGE_TOKENS;
  p->n_planes = n_planes;
  profile_kinds(desc->profile, &p->kind_k, &p->kind_v);
  for (int i = 0; i < 4; ++i) p->plane[i] = g[i];
  p->ptrs.assign(planes, planes + desc->num_layers * n_planes);
  cudaError_t e = cudaGetDevice(&p->device);
  if (e != cudaSuccess) {
    delete p;
    return cuda_fail(e, "cudaGetDevice");
  }
  p->num_sms = device_sm_count(p->device);
  p->status = status_word();
  if (!p->status || !p->num_sms) {
    delete p;
    return fail(NK_ERR_CUDA, "device query failed (status word / SM count)");
  }
  p->tmap.resize(static_cast<size_t>(desc->num_layers) * 2);
  for (int l = 0; l < desc->num_layers; ++l) {
    for (int s = 0; s < 2; ++s) {
      rc = encode_code_tmap(&p->tmap[l * 2 + s], p->ptrs[l * n_planes + s], g[s].row_bytes, rows);
      if (rc) {
        delete p;
        return rc;
      }
    }
  }
  *out = p;
  return NK_OK;
}

extern "C" int nk_pool_destroy(nk_pool* pool) {
  clear_error();
  delete pool;
  return NK_OK;
}

extern "C" int nk_page_copy_columns(const nk_pool* pool, int32_t src, int32_t dst, int32_t ncols,
                                    void* stream) {
  clear_error();
  if (!pool) return fail(NK_ERR_INVALID_ARG, "pool is NULL");
  if (src < 0 || src >= pool->M || dst < 0 || dst >= pool->M || src == dst)
    return fail(NK_ERR_RANGE, "src/dst page groups must be distinct and in [0, M)");
  if (ncols < 0 || ncols > NK_PAGE_TOKENS) return fail(NK_ERR_SHAPE, "ncols must be in [0, 64]");
  if (ncols == 0) return NK_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int H = pool->desc.num_kv_heads;
  for (int l = 0; l < pool->desc.num_layers; ++l) {
    for (int i = 0; i < pool->n_planes; ++i) {
      const size_t rb = pool->plane[i].row_bytes;
      const int hm = pool->desc.order == NK_HEAD_MAJOR;
      // columns [0, ncols) of every head are one contiguous run per head; the
      // heads of a page group are tile_row(g, 1) - tile_row(g, 0) rows apart
      const size_t head_pitch = static_cast<size_t>(tile_row(0, 1, H, pool->M, hm)) * rb;
      char* base = static_cast<char*>(pool->ptrs[l * pool->n_planes + i]);
      cudaError_t e = cudaMemcpy2DAsync(base + tile_row(dst, 0, H, pool->M, hm) * rb, head_pitch,
                                        base + tile_row(src, 0, H, pool->M, hm) * rb, head_pitch, rb * ncols, H,
                                        cudaMemcpyDeviceToDevice, s);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync (page copy)");
    }
  }
  return NK_OK;
}

extern "C" int nk_status_read(int32_t* status, int32_t clear, void* stream) {
  clear_error();
  if (!status) return fail(NK_ERR_INVALID_ARG, "status is NULL");
  int* dev = status_word();
  if (!dev) return fail(NK_ERR_CUDA, "status word address unavailable");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, dev, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(dev, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *status = v;
  return NK_OK;
}
