// Diagnostic kernel for the bounded-wait failure path: one thread waits on an
// mbarrier phase that nothing completes, through the same bounded wait the
// attention pipeline uses, and reports the expiry in a status word.
#include "hpa_internal.cuh"

namespace hpa {
namespace {

__global__ void selftest_wait_kernel(int32_t *status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(b, 0, limit_ns))
    atomicOr(reinterpret_cast<int *>(status), HPA_STATUS_TIMEOUT);
}

}  // namespace

cudaError_t launch_selftest_wait(int32_t *status, long long limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, static_cast<unsigned long long>(limit_ns));
  return cudaGetLastError();
}

}  // namespace hpa
