// q3a_selftest.cu — q3a_selftest_bounded_wait: one block that waits on an
// mbarrier through the same bounded-wait routine every kernel of the library
// uses, so the timeout path (error word set, wait abandoned, kernel returns)
// can be exercised on a GPU without faulting or hanging it.
//
// With arrive == 0 nothing ever arrives on the barrier: the wait gives up after
// `limit_cycles` SM cycles, records kDevTimeoutSelftest in the error word and
// the kernel returns normally; q3a_last_device_error then reports
// Q3A_ETIMEOUT. With arrive != 0 thread 0 arrives first and the wait returns
// at once, leaving the word at zero.
#include "q3a.h"
#include "q3a_device.cuh"
#include "q3a_internal.h"

namespace q3a {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint32_t* err,
                                                                   long long limit_cycles,
                                                                   int arrive) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();  // barrier initialised
  if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
  mbar_wait(&bar, 0, err, kDevTimeoutSelftest, &abort_flag, limit_cycles);
}

}  // namespace
}  // namespace q3a

using namespace q3a;

extern "C" q3a_status q3a_selftest_bounded_wait(void* workspace, size_t ws_bytes,
                                                long long limit_cycles, int arrive,
                                                void* stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u) || ws_bytes < 256)
    return Q3A_EINVAL;
  if (limit_cycles <= 0 || limit_cycles > kWaitLimitCycles) return Q3A_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = static_cast<uint32_t*>(workspace);
  if (cudaMemsetAsync(err, 0, sizeof(uint32_t), st) != cudaSuccess) return Q3A_ECUDA;
  bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_cycles, arrive);
  return cudaGetLastError() == cudaSuccess ? Q3A_OK : Q3A_ECUDA;
}
