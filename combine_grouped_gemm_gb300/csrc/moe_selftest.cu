// moe_selftest_wait: exercises the bounded waits every kernel of this library uses (a wait that
// runs out records MOE_DEV_TIMEOUT in the workspace status word and raises the CTA's abort
// flag, on which the CTA's other waits return at once), without any real work that could go
// wrong: the barriers waited on are simply never completed.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);   // nothing ever arrives on either barrier
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  if (threadIdx.x == 0) {
    (void)mbar_wait(&bars[0], 0, abort, status, limit_ns);
  } else if (threadIdx.x == 32) {
    // returns when the first wait raises the abort flag (or, should that fail, after 3 x limit)
    (void)mbar_wait(&bars[1], 0, abort, status, 3 * limit_ns);
  }
  __syncthreads();
}

}  // namespace
}  // namespace moe

extern "C" int moe_selftest_wait(void* ws, int64_t limit_ns, cudaStream_t stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 15u)) return MOE_ERR_INVALID_ARG;
  if (limit_ns < 1000 || limit_ns > 10000000000LL) return MOE_ERR_INVALID_ARG;
  moe::selftest_wait_kernel<<<1, 64, 0, stream>>>(static_cast<uint32_t*>(ws),
                                                 static_cast<uint64_t>(limit_ns));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(e);
}
