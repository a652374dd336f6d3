// internal.h -- host-side pool handle and helpers shared by the libnk
// translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "nk.h"

namespace nk {

// Vector codec of one side (K or V) of a profile.
enum Kind : int { KIND_BF16 = 0, KIND_INT8 = 1, KIND_FP8 = 2, KIND_NVFP4 = 3 };

struct PlaneGeom {
  int elem_bytes;  // bytes per element
  int X;           // leading extent (elements per token per head)
  int row_bytes;   // X * elem_bytes: bytes per token per head
};

}  // namespace nk

struct nk_pool {
  nk_pool_desc desc;
  int32_t M;              // physical page groups
  int32_t L;              // logical pages per table row = ceil(S / 64)
  int n_planes;           // 2 (BF16) or 4
  nk::Kind kind_k, kind_v;
  nk::PlaneGeom plane[4];  // [K code, V code, K scale, V scale]
  std::vector<void*> ptrs;            // [layer * n_planes + i]
  std::vector<CUtensorMap> tmap;      // [layer * 2 + {0: K code, 1: V code}]
  int device;
  int num_sms;
  int* status;            // device address of the status word of `device`
};

namespace nk {

// Thread-local error text; returns `code` for convenient `return fail(...)`.
int fail(int code, const std::string& msg);
int cuda_fail(cudaError_t e, const char* what);
void clear_error();

int profile_kinds(int profile, Kind* k, Kind* v);
int plane_geoms(int profile, int D, int* n_planes, PlaneGeom g[4]);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// First row (of row_bytes each) of the 64-token tile of page group g, KV head
// h in a plane ("Paged KV cache" page, closed plane orders): page-major
// [X, P, H, M] gives (g * H + h) * 64, head-major [X, P, M, H] (h * M + g) * 64.
__host__ __device__ __forceinline__ int64_t tile_row(int g, int h, int H, int M, int head_major) {
  return head_major ? (static_cast<int64_t>(h) * M + g) * 64 : (static_cast<int64_t>(g) * H + h) * 64;
}

// Caches the SM count of a device.
int device_sm_count(int device);

// Device address of the status word on the current device (nullptr on error).
int* status_word();

// 2-D TMA descriptor over `rows` rows of `row_bytes` bytes (viewed as uint8):
// boxes of 64 rows x min(row_bytes, 128) bytes with the matching swizzle.
int encode_code_tmap(CUtensorMap* m, void* base, int row_bytes, int64_t rows);

}  // namespace nk
