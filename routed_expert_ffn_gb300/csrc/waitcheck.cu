// Check of the bounded device waits the pipelined kernels rely on: one
// thread waits on a shared-memory mbarrier that nothing arrives on, with the
// same bounded wait the GEMM and router pipelines use.  The wait gives up
// after kWaitLimitNs, raises the CTA's abort flag and latches
// kStatusTimeoutCheck in the workspace status word; the kernel then returns,
// so the context stays usable.  No fault, trap or unbounded spin is involved.
#include "moe_internal.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(32) bounded_wait_check_kernel(uint32_t *__restrict__ status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    // phase 0 never completes: no thread arrives
    mbar_wait(&bar, 0u, reinterpret_cast<volatile int *>(&abort_flag), status,
              kStatusTimeoutCheck);
  }
}

}  // namespace

cudaError_t launch_bounded_wait_check(uint32_t *status, cudaStream_t s) {
  bounded_wait_check_kernel<<<1, 32, 0, s>>>(status);
  return cudaGetLastError();
}

}  // namespace moe
