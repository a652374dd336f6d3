// decode_noalloc.cu -- paged decode attention that allocates nothing.
//
// Some callers cannot call cudaMalloc: code that runs inside an allocator's
// own callbacks, a host runtime that forbids device allocation once its
// memory budget is fixed at start-up, or a serving loop that must never
// block on the driver's allocator.  For them this entry point keeps the
// split-K partials of nk_paged_decode_attention in a file-scope static device
// array of NK_NOALLOC_SCRATCH_BYTES bytes.  The driver reserves that array
// when this module is loaded on a device, and it stays reserved on every
// device that loaded it until the process exits.
//
// The array's host-side name is only a stand-in for the symbol, not a device
// address: a kernel given it would fault, or silently use the wrong memory
// where the GPU can reach host memory.  So the first call on a device, with
// that device current, asks the runtime for the array's device address with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture.  The cached address lives as long as the process: after a reset
// of the device's primary context (cudaDeviceReset) the module is loaded
// again and the cached address is stale, so the entry point must not be used
// across such a reset.  All calls share the array and it keeps the last
// call's contents; every slot of split partials a call reads it wrote first,
// so nothing needs clearing.  Two calls that overlap on the GPU race on the
// array.
#include <mutex>

#include "internal.h"

namespace nk {
int decode_with_scratch(const void* q, int32_t Hq, const nk_pool* pool, int32_t layer,
                        const int32_t* block_tables, const int32_t* table_rows,
                        const int32_t* frontiers, int32_t B, int32_t T, float softmax_scale,
                        void* out, float* lse, void* scratch, size_t max_ws, cudaStream_t s);
}  // namespace nk

using namespace nk;

static __device__ __align__(256) unsigned char g_decode_scratch[NK_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on `device` (which must be current);
// set up once per device.
static int scratch_address(int device, void** out) {
  static std::mutex mu;
  static void* cache[64] = {nullptr};
  if (device < 0 || device >= 64) return fail(NK_ERR_INVALID_ARG, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress (static decode scratch)");
    cache[device] = p;
  }
  *out = cache[device];
  return NK_OK;
}

extern "C" int nk_paged_decode_attention_noalloc(const void* q, int32_t Hq, const nk_pool* pool,
                                                 int32_t layer, const int32_t* block_tables,
                                                 const int32_t* table_rows,
                                                 const int32_t* frontiers, int32_t B, int32_t T,
                                                 float softmax_scale, void* out, float* lse,
                                                 void* stream) {
  clear_error();
  if (!pool) return fail(NK_ERR_INVALID_ARG, "pool is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != pool->device) return fail(NK_ERR_INVALID_ARG, "make the pool's device current first");
  void* scratch = nullptr;
  int rc = scratch_address(dev, &scratch);
  if (rc) return rc;
  return decode_with_scratch(q, Hq, pool, layer, block_tables, table_rows, frontiers, B, T,
                             softmax_scale, out, lse, scratch, NK_NOALLOC_SCRATCH_BYTES,
                             static_cast<cudaStream_t>(stream));
}
