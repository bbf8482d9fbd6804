// attn_selftest.cu - exercises the kernels' bounded-wait failure path on the
// GPU without faulting it: one thread waits, with a short limit, on an
// mbarrier phase that nothing completes. When the limit expires it records
// STATUS_TIMEOUT in the device status word exactly as a stuck attention CTA
// would, and returns normally, leaving the context usable.
#include "params.h"
#include "ptx.cuh"

namespace attn {

__global__ void wait_timeout_probe_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // expects one arrival; none is ever made
    mbar_init_fence();
    if (!mbar_wait_for(b, 0, limit_ns) && status) atomicOr(status, STATUS_TIMEOUT);
  }
}

cudaError_t launch_wait_timeout_probe(int* status, unsigned long long limit_ns,
                                      cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace attn
