// Self-test of the bounded mbarrier wait that every pipelined kernel of the
// library uses (the write kernel's stage barriers, the prefill's hand-offs):
// one warp waits on a barrier that nothing arrives at, gives up after the
// given number of attempts, reports KV_INT4_DEV_TIMEOUT and returns.  It
// exercises the time-out path on a GPU without a fault or a hang, and its
// cycle count bounds how long the kernels' own limit (kMaxWaitIters
// attempts) can hold a warp.

#include <cuda_runtime.h>

#include "../../include/kvint4.h"
#include "common.cuh"
#include "internal.h"

namespace kvint4 {

__global__ void __launch_bounds__(32) selftest_wait_kernel(int iterations, int32_t* status,
                                                           unsigned long long* cycles) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const long long t0 = clock64();
  bool done = false;
  for (int n = 0; n < iterations && !done; n++) done = mbar_try_wait(b, 0);  // phase 0 never completes
  const long long t1 = clock64();
  if (threadIdx.x == 0) {
    if (!done) flag(status, KV_INT4_DEV_TIMEOUT);
    if (cycles) *cycles = (unsigned long long)(t1 - t0);
  }
}

}  // namespace kvint4

extern "C" KVINT4_API int kv_int4_selftest_wait(int iterations, int32_t* dev_status, uint64_t* dev_cycles,
                                                void* stream) {
  if (iterations < 0) return KV_INT4_ERR_SIZE;
  if (!dev_status) return KV_INT4_ERR_NULL;
  kvint4::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(iterations, dev_status,
                                                    reinterpret_cast<unsigned long long*>(dev_cycles));
  return cudaGetLastError() == cudaSuccess ? KV_INT4_OK : KV_INT4_ERR_CUDA;
}
