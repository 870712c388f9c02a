// selftest.cu -- failure detection without a GPU fault: a kernel whose bounded
// waits nothing can satisfy, so that a test can watch them give up.  The
// kernel waits on an mbarrier no thread arrives on (the wait every TMA and
// tensor-core pipeline of the library uses) and on a global word no one writes
// (the wait of a CTA for another), each with the caller's limit.  Each wait
// raises DFLASH2_DEVERR_TIMEOUT in the error word and the kernel returns
// normally, leaving the context usable.
#include "common.cuh"
#include "launch.h"

namespace dflash2 {
namespace {

__global__ void wait_timeout_kernel(const uint32_t* flag, uint64_t limit_ns, uint32_t* err, uint32_t* result) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool arrived = mbar_wait_bounded(&bar, 0, err, limit_ns);   // no thread arrives
    const bool written = flag_wait_bounded(flag, 1u, err, limit_ns);  // no one writes 1
    // bit 0 / 1: a wait succeeded (never); bit 2: the kernel reached its end
    *result = (arrived ? 1u : 0u) | (written ? 2u : 0u) | 4u;
  }
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(const uint32_t* flag, uint64_t limit_ns, uint32_t* err, uint32_t* result,
                                         cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(flag, limit_ns, err, result);
  return cudaGetLastError();
}

}  // namespace dflash2
