// decode_nvfp4.cu -- paged decode attention instantiations of the NVFP4-G16 profile.
#include "decode.cuh"

namespace nk {

cudaError_t decode_nvfp4(const nk_pool* p, int layer, const DecodeArgs& a, int nqt, dim3 grid,
                      cudaStream_t s) {
  return decode_dispatch<KIND_NVFP4, KIND_NVFP4>(p, layer, a, nqt, grid, s);
}

int occupancy_nvfp4(int D, int nqt, int* ring_bytes) { return decode_occupancy<KIND_NVFP4, KIND_NVFP4>(D, nqt, ring_bytes); }

}  // namespace nk
