// Self-test of the bounded pipeline wait every kernel of this library uses:
// one warp waits on an mbarrier that nothing ever arrives on, with a short
// time limit; a second warp waits on another such barrier with the kernels'
// full limit and must leave as soon as the first has raised the shared abort
// flag.  Nothing faults or hangs: both waits end, and the kernel reports the
// status code and both wait durations.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace diffattn {
namespace {

constexpr uint64_t FULL_TIMEOUT_NS = 2000000000ull;

__global__ void __launch_bounds__(64) diffattn_selftest_wait_kernel(int32_t *status,
                                                                    uint64_t timeout_ns) {
  __shared__ uint64_t never[2];
  __shared__ int abort_flag;
  __shared__ uint64_t waited_ns[2];
  __shared__ int timed_out;
  if (threadIdx.x == 0) {
    mbar_init(&never[0], 1);
    mbar_init(&never[1], 1);
    abort_flag = 0;
    timed_out = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x / 32;
  if ((threadIdx.x & 31) == 0) {
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait(&never[warp], 0, &abort_flag, warp == 0 ? timeout_ns : FULL_TIMEOUT_NS);
    waited_ns[warp] = globaltimer_ns() - t0;
    if (!ok && warp == 0) timed_out = 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    status[1] = static_cast<int32_t>(waited_ns[0] / 1000);  // microseconds
    status[2] = static_cast<int32_t>(waited_ns[1] / 1000);
    status[0] = timed_out && abort_flag ? static_cast<int32_t>(DIFFATTN_ERR_TIMEOUT) : 0;
  }
}

}  // namespace

diffattn_status launch_selftest_wait(int32_t *status, int64_t timeout_ns, cudaStream_t stream) {
  diffattn_selftest_wait_kernel<<<1, 64, 0, stream>>>(status, static_cast<uint64_t>(timeout_ns));
  return cudaGetLastError() == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

}  // namespace diffattn
