// pa_check_wait_limit: a diagnostic of the bounded mbarrier waits that every
// kernel of the library uses, run where nothing ever completes the barriers.
//
// Each wait polls its barrier and reads the global timer; past its limit it
// raises the CTA's abort flag, records the timeout bit in the device error
// word and returns, and the other warps of the CTA return as soon as they see
// the flag. This kernel runs exactly that code with two warps on two barriers
// that no thread or copy ever arrives on.
#include <cstdint>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Warp 0 gives up after limit_ns; warp 1, whose own limit is 50 times longer,
// must leave through the abort flag that warp 0 raises.
__global__ void __launch_bounds__(64) wait_limit_kernel(unsigned long long limit_ns, unsigned* err) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  mbar_wait_bounded(&bars[warp], 0, &abort_flag, err, warp == 0 ? limit_ns : 50ull * limit_ns);
  __syncwarp();
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_check_wait_limit(uint64_t limit_ns, cudaStream_t stream) {
  if (limit_ns < 1000ull || limit_ns > 100000000ull) return PA_ERR_INVALID_ARG;
  unsigned* err = nullptr;
  int sms = 0;
  const pa_status s = pa::device_state(&err, &sms);
  if (s != PA_OK) return s;
  pa::wait_limit_kernel<<<1, 64, 0, stream>>>((unsigned long long)limit_ns, err);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
