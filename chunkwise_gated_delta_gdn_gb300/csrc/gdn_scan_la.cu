// gdn_scan_la.cu -- the scan kernel of the bf16 scalar-gate (GDN) path: one
// CTA of 384 threads per (sequence, value head, 64-column dv slice), running
// the block of gdn_scan_la.cuh after the prep kernel has written every image.
#include "gdn_scan_la.cuh"

namespace gdn {
namespace {

using namespace sm100;

template <int C, int DK>
__global__ void __launch_bounds__(kThreads, 1)
gdn_scan_la_kernel(const ScanArgs a, const __grid_constant__ ScanMaps maps) {
  using SM = LaSmem<C, DK>;
  extern __shared__ unsigned char smem_raw[];
  // 1 KB-aligned base, as an offset into the shared array (the compiler then
  // knows every access below is to shared memory)
  unsigned char *sm = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
  if (sm - smem_raw > SM::kSlack) {  // dynamic shared memory not aligned as needed
    if (threadIdx.x == 0) atomicOr(a.flags, kFlagLaunchConfig);
    return;
  }
  scan_la_block<C, DK>(a, maps, blockIdx.x, sm, nullptr);
}

template <int C, int DK>
cudaError_t launch_one(const ScanArgs &a, const ScanMaps &maps, cudaStream_t stream) {
  using SM = LaSmem<C, DK>;
  auto kern = gdn_scan_la_kernel<C, DK>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (err != cudaSuccess) return err;
  const long blocks = (long)a.seq.n_seqs * a.HV * (a.dv / NS);
  if (blocks > 0x7fffffffL) return cudaErrorInvalidValue;
  kern<<<(unsigned)blocks, kThreads, SM::kBytes, stream>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_la(const ScanArgs &a, const ScanMaps &maps, int chunk, int dk,
                           cudaStream_t stream) {
  if (chunk == 64 && dk == 128) return launch_one<64, 128>(a, maps, stream);
  if (chunk == 64 && dk == 64) return launch_one<64, 64>(a, maps, stream);
  if (chunk == 32 && dk == 128) return launch_one<32, 128>(a, maps, stream);
  if (chunk == 32 && dk == 64) return launch_one<32, 64>(a, maps, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
