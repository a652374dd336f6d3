// selftest.cu -- a kernel whose bounded wait is made to run out, so that the
// timeout path every pipeline wait relies on (mbar_wait_bounded: give up
// after a wall-clock limit, record NK_STATUS_TIMEOUT, return) can be checked
// on a GPU without any fault or hang.
//
// One thread arms an mbarrier that expects two arrivals and arrives once, so
// the phase can never complete; no copy or other thread is involved.  The
// wait gives up after `limit_us` microseconds and the kernel returns
// normally: the context stays usable and the status word tells the host.
#include "device.cuh"
#include "internal.h"

namespace nk {

__global__ void bounded_wait_selftest_kernel(int* status, uint64_t limit_ns, long long* waited_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 2);
  fence_barrier_init();
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar)) : "memory");
  const uint64_t t0 = globaltimer_ns();
  const bool done = mbar_wait_bounded(&bar, 0, status, limit_ns);
  const uint64_t t1 = globaltimer_ns();
  if (waited_ns) *waited_ns = done ? -1 : static_cast<long long>(t1 - t0);
}

}  // namespace nk

using namespace nk;

extern "C" int nk_selftest_bounded_wait(int32_t limit_us, long long* waited_ns, void* stream) {
  clear_error();
  if (limit_us < 1 || limit_us > 1000000)
    return fail(NK_ERR_INVALID_ARG, "limit_us must be in [1, 1000000]");
  int* st = status_word();
  if (!st) return fail(NK_ERR_CUDA, "status word address unavailable");
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      st, static_cast<uint64_t>(limit_us) * 1000ull, waited_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return NK_OK;
}
