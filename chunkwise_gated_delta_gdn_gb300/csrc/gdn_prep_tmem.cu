// gdn_prep_tmem.cu -- the chunk-prep kernel of the bf16 scalar-gate (GDN)
// path: one CTA of 128 threads per (chunk slot, q/k head), running the unit of
// gdn_prep_tmem.cuh.  Four CTAs share an SM (128 tensor-memory columns, about
// 56 KB of shared memory and at most 128 registers a thread each), so that
// their latency-bound phases overlap.  Launched over every slot before the
// scan kernel, or over the first slots only, publishing each unit's ready
// flag, ahead of the lockstep launch (gdn_lockstep.cu).
#include "gdn_prep_tmem.cuh"

namespace gdn {
namespace {

using namespace sm100;

template <int C, int DK>
__global__ void __launch_bounds__(128, 4)
gdn_prep_tmem_kernel(const PrepArgs a, const __grid_constant__ ScanMaps maps, int *ready) {
  extern __shared__ unsigned char smem_raw[];
  // 1 KB-aligned base, as an offset into the shared array (the compiler then
  // knows every access below is to shared memory)
  unsigned char *sm = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + PrepTmemSmem<C>::kMisc);
  constexpr uint32_t kCols = 128;
  if (threadIdx.x < 32) tmem_alloc(smem_addr(tslot), kCols);
  if (threadIdx.x == 0) prep_tmem_init_barriers<C>(sm);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tslot;
  PrepPhases ph;
  prep_tmem_unit<C, DK>(a, maps, blockIdx.x, blockIdx.y, sm, tmem, threadIdx.x, 1, ready, ph);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (threadIdx.x < 32) tmem_dealloc(tmem, kCols);
}

template <int C, int DK>
cudaError_t launch_one(const PrepArgs &a, const ScanMaps &maps, int n_slots, int *ready,
                       cudaStream_t stream) {
  using SM = PrepTmemSmem<C>;
  auto kern = gdn_prep_tmem_kernel<C, DK>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (err != cudaSuccess) return err;
  // four CTAs per SM need the largest shared-memory carve-out
  err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (err != cudaSuccess) return err;
  kern<<<dim3(n_slots, a.H), 128, SM::kBytes, stream>>>(a, maps, ready);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_tmem(const PrepArgs &a, const ScanMaps &maps, int chunk, int dk,
                             cudaStream_t stream, int n_slots, int *ready) {
  if (n_slots < 0) n_slots = a.n_slots;
  if (n_slots == 0) return cudaSuccess;
  if (chunk == 64 && dk == 128) return launch_one<64, 128>(a, maps, n_slots, ready, stream);
  if (chunk == 64 && dk == 64) return launch_one<64, 64>(a, maps, n_slots, ready, stream);
  if (chunk == 32 && dk == 128) return launch_one<32, 128>(a, maps, n_slots, ready, stream);
  if (chunk == 32 && dk == 64) return launch_one<32, 64>(a, maps, n_slots, ready, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
