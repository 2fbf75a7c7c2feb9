// Self-test of the device-side wait bound: one warp waits on an mbarrier
// phase that nothing completes; the wait must give up, record
// kDevTimeoutSelfTest in the error word and let the kernel exit, leaving the
// context usable.
#include "moe.h"
#include "ptx.cuh"

namespace {

__global__ void selftest_timeout_kernel(int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    moe::ptx::mbar_init(&bar, 1);
    moe::ptx::fence_barrier_init();
  }
  __syncthreads();
  // no thread ever arrives on `bar`: phase 0 never completes
  if (!moe::ptx::mbar_wait(&bar, 0, nullptr)) {
    if (threadIdx.x == 0) moe::set_error(err, moe::kDevTimeoutSelfTest);
  }
}

}  // namespace

extern "C" moe_status moe_selftest_timeout(void* ws, moe_stream_t stream) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 15u)) return MOE_ERR_INVALID_ARG;
  selftest_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<int*>(ws));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
