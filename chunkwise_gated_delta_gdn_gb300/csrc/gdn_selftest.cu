// gdn_selftest.cu -- self-test of the bounded waits of the tensor-core kernels.
//
// Every wait of the prep and scan kernels on an mbarrier (a TMA load, a bulk
// copy or a tensor-core product completing) gives up after a clock budget:
// it sets the kernel's abort flag, every later wait returns at once, the
// kernel finishes with the same control flow in every thread and sets the
// TIMEOUT bit of the device status word.  A completion that never comes thus
// ends as a status the host reads, not as a hung GPU.  This kernel runs that
// same wait (sm100::mbar_wait) on a barrier of its own:
//   complete = 0: nothing ever arrives, so every wait must run out of its
//                 budget and the status word must read TIMEOUT;
//   complete = 1: one thread arrives first, so the phase completes and the
//                 waits must return with no flag set.
// Nothing faults and nothing spins past the budget either way.
#include <stdint.h>

#include "gdn.h"
#include "gdn_internal.h"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

__global__ void __launch_bounds__(32) gdn_wait_selftest_kernel(uint32_t *flags, long long budget,
                                                              int complete) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  const uint32_t b = sm100::smem_addr(&bar);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    sm100::mbar_init(b, 1);
    sm100::mbar_fence_init();
  }
  __syncthreads();
  if (complete && threadIdx.x == 0) sm100::mbar_arrive(b);
  sm100::mbar_wait(b, 0, &abort_flag, budget);
  __syncthreads();
  if (threadIdx.x == 0 && abort_flag) atomicOr(flags, kFlagTimeout);
}

}  // namespace
}  // namespace gdn

extern "C" {

gdn_status gdn_selftest_wait(uint32_t *flags, long long budget_cycles, int complete,
                             gdn_stream_t stream_) {
  if (!flags || (reinterpret_cast<uintptr_t>(flags) & 3u) != 0) return GDN_ERR_INVALID_ARG;
  if (budget_cycles <= 0 || budget_cycles > 4000000000LL) return GDN_ERR_INVALID_ARG;
  if (complete != 0 && complete != 1) return GDN_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaMemsetAsync(flags, 0, sizeof(uint32_t), stream) != cudaSuccess) return GDN_ERR_CUDA;
  gdn::gdn_wait_selftest_kernel<<<1, 32, 0, stream>>>(flags, budget_cycles, complete);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // extern "C"
