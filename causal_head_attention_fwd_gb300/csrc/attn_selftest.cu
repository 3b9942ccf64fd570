// Failure-detection self-test: one warp waits, with the same bounded-wait
// mechanism the attention kernels use (mbarrier try_wait polled against
// %globaltimer), on a barrier phase that nothing will ever complete. When its
// limit passes it records ATTN_ERR_TIMEOUT in the device error word and
// returns, exactly as a kernel whose producer died would, so the host-side
// reporting path can be tested without faulting or hanging the GPU.
#include "../../include/attn.h"
#include "common.cuh"

namespace attn {

__global__ void attn_selftest_timeout_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t never;              // initialised with one expected arrival; none comes
  __shared__ volatile int abort_sh;
  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&never, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint32_t a = smem_u32(&never);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, 0)) {
    if (abort_sh) break;
    if (globaltimer_ns() - t0 > limit_ns) {
      abort_sh = 1;
      atomicCAS(err, 0, (int)ATTN_ERR_TIMEOUT);
      break;
    }
  }
}

}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 10000000u) return ATTN_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (!err) return ATTN_ERR_CUDA;
  attn_selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      err, (unsigned long long)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
