// selftest.cu -- exercises the bounded-wait error path of the tensor-core
// kernels without faulting or hanging the GPU.
#include "kernels.h"
#include "tc.cuh"

namespace la {
namespace {

// One thread initialises an mbarrier expecting one arrival.  With `arrive`
// set it arrives itself and the wait completes at once; otherwise nothing
// ever arrives and the wait gives up after limit_ns, setting the status word.
__global__ void bounded_wait_kernel(int arrive, uint64_t limit_ns, unsigned* status) {
  __shared__ uint64_t bar;
  const uint32_t b = tc::smem_u32(&bar);
  tc::mbar_init(b, 1);
  tc::fence_mbar_init();
  if (arrive) tc::mbar_arrive(b);
  tc::mbar_wait_ns(b, 0, status, limit_ns);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int arrive, uint64_t limit_ns, unsigned* status, cudaStream_t stream) {
  bounded_wait_kernel<<<1, 1, 0, stream>>>(arrive, limit_ns, status);
  return cudaGetLastError();
}

}  // namespace la
