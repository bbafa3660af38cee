// selftest.cu -- exercises the bounded mbarrier wait that every kernel of
// the library uses, on a barrier that nothing arrives on: the wait gives up
// after the given time, records PKV_EDEV_TIMEOUT in the device error word
// and the kernel returns, leaving the context usable.  Not part of the
// attention path; it lets a test check the failure path on a GPU without
// faulting or hanging it.
#include "common.cuh"
#include "kernels.h"
#include "tc5.cuh"

namespace pkv {

namespace {

__global__ void bounded_wait_selftest_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_word;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    tc5::mbar_init(b, 1);
    abort_word = 0;
    tc5::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 never completes: nothing arrives on the barrier
    tc5::mbar_wait_for(b, 0, &abort_word, err, limit_ns, /*honor_abort=*/false);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int* err, uint64_t limit_ns,
                                         cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace pkv
