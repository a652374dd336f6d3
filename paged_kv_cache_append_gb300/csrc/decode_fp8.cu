// decode_fp8.cu -- paged decode attention instantiations of the FP8-E4M3FN-row256 profile.
#include "decode.cuh"

namespace nk {

cudaError_t decode_fp8(const nk_pool* p, int layer, const DecodeArgs& a, int nqt, dim3 grid,
                      cudaStream_t s) {
  return decode_dispatch<KIND_FP8, KIND_FP8>(p, layer, a, nqt, grid, s);
}

int occupancy_fp8(int D, int nqt, int* ring_bytes) { return decode_occupancy<KIND_FP8, KIND_FP8>(D, nqt, ring_bytes); }

}  // namespace nk
