// prefill.cu -- chunked prefill / replay attention through the block tables.
#include "internal.h"

using namespace nk;

extern "C" int nk_prefill_workspace_bytes(const nk_pool* pool, int32_t B, int32_t Tc, int32_t Hq,
                                          size_t* bytes) {
  clear_error();
  if (!pool || !bytes) return fail(NK_ERR_INVALID_ARG, "null argument");
  *bytes = 0;
  return NK_OK;
}

extern "C" int nk_paged_prefill_attention(const void*, int32_t, const nk_pool*, int32_t,
                                          const int32_t*, const int32_t*, const int32_t*,
                                          const int32_t*, int32_t, int32_t, float, void*, float*,
                                          void*, size_t, void*) {
  clear_error();
  return fail(NK_ERR_UNSUPPORTED, "chunked prefill is not built yet");
}
