// decode_k8v4.cu -- paged decode attention instantiations of the K8V4 profile.
#include "decode.cuh"

namespace nk {

cudaError_t decode_k8v4(const nk_pool* p, int layer, const DecodeArgs& a, int nqt, dim3 grid,
                      cudaStream_t s) {
  return decode_dispatch<KIND_FP8, KIND_NVFP4>(p, layer, a, nqt, grid, s);
}

int occupancy_k8v4(int D, int nqt, int* ring_bytes) { return decode_occupancy<KIND_FP8, KIND_NVFP4>(D, nqt, ring_bytes); }

}  // namespace nk
