// decode_bf16.cu -- paged decode attention instantiations of the BF16 profile.
#include "decode.cuh"

namespace nk {

cudaError_t decode_bf16(const nk_pool* p, int layer, const DecodeArgs& a, int nqt, dim3 grid,
                      cudaStream_t s) {
  return decode_dispatch<KIND_BF16, KIND_BF16>(p, layer, a, nqt, grid, s);
}

int occupancy_bf16(int D, int nqt, int* ring_bytes) { return decode_occupancy<KIND_BF16, KIND_BF16>(D, nqt, ring_bytes); }

}  // namespace nk
