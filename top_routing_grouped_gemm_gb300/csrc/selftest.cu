// Self-test of the bounded device waits that every pipelined kernel of the library uses.
#include "ptx.cuh"

namespace {

// One thread waits, with the library's bounded wait, on an mbarrier that nothing will ever
// arrive on; when the limit runs out it reports MOE_ERR_TIMEOUT and returns.  The kernel
// always ends after about timeout_ns: it can neither hang nor fault.
__global__ void wait_timeout_kernel(int32_t* dev_status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int no_abort;
  if (threadIdx.x == 0) {
    moe::mbar_init(&bar, 1);
    no_abort = 0;
    moe::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!moe::mbar_wait(&bar, 0, reinterpret_cast<volatile int*>(&no_abort), timeout_ns))
      moe::report_status(dev_status, MOE_ERR_TIMEOUT);
  }
}

}  // namespace

extern "C" int moe_selftest_wait_timeout(int32_t* dev_status, int32_t timeout_ms,
                                         moe_stream_t stream) {
  if (!dev_status || timeout_ms <= 0 || timeout_ms > 2000) return MOE_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, stream>>>(dev_status,
                                            static_cast<uint64_t>(timeout_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
