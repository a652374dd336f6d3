// decode_int8.cu -- paged decode attention instantiations of the INT8-G64 profile.
#include "decode.cuh"

namespace nk {

cudaError_t decode_int8(const nk_pool* p, int layer, const DecodeArgs& a, int nqt, dim3 grid,
                      cudaStream_t s) {
  return decode_dispatch<KIND_INT8, KIND_INT8>(p, layer, a, nqt, grid, s);
}

int occupancy_int8(int D, int nqt, int* ring_bytes) { return decode_occupancy<KIND_INT8, KIND_INT8>(D, nqt, ring_bytes); }

}  // namespace nk
