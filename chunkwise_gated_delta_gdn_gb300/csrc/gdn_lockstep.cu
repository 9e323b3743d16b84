// gdn_lockstep.cu -- the chunk prep and the scan of the bf16 scalar-gate (GDN)
// path in one launch, in lockstep (the fused prep + scan composition of
// ROCm/rocm-libraries PR #11223, "Summary", in a form for this GPU).
//
// The grid is cooperative, so that every CTA is resident at once.  Its first
// n_scan CTAs are the scan's blocks (gdn_scan_la.cuh, unchanged arithmetic);
// the others run the prep (gdn_prep_tmem.cuh, unchanged arithmetic) in three
// persistent warpgroups each, over the (chunk slot, q/k head) units in chunk
// order.  A warpgroup that finishes a unit waits for its bulk stores to
// complete and sets that unit's ready flag (release, gpu scope); the scan loads
// a prep image only once its flag is set (acquire, bounded wait).  The prep
// never waits for the scan, so the scan always makes progress, and the images
// of a chunk are read back soon after they are written.
//
// Both halves run the same device code as the split kernels, on the same
// inputs, so the results equal gdn_chunk_fwd's bit for bit.  The prep has only
// the SMs the scan leaves (one CTA per SM: the scan needs about 213 KB of
// shared memory), three warpgroups each: fewer units in flight than the split
// prep kernel's four CTAs on every SM.  So the prep gets a head start: the
// split prep kernel runs first over the first head_slots chunk slots on every
// SM, setting their flags as well, and the lockstep's prep warpgroups take the
// slots after them while the scan walks the chunks.
#include "gdn_prep_tmem.cuh"
#include "gdn_scan_la.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kPrepGroups = 3;  // prep warpgroups per prep CTA

template <int C, int DK>
struct LockSmem {
  static constexpr int kScan = LaSmem<C, DK>::kUsed;
  static constexpr int kPrep = kPrepGroups * PrepTmemSmem<C>::kSlice;
  static constexpr int kUsed = kScan > kPrep ? kScan : kPrep;
  static constexpr int kBytes = kUsed + 1024;  // alignment slack
  static_assert(kThreads >= kPrepGroups * 128, "prep warpgroups of one CTA");
  static_assert(kBytes <= 232448, "shared memory of one CTA");
};

template <int C, int DK>
__global__ void __launch_bounds__(kThreads, 1)
gdn_lockstep_kernel(const PrepArgs pa, const ScanArgs sa, const __grid_constant__ ScanMaps maps,
                    int n_scan, int *ready, int unit0) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
  if (blockIdx.x < (unsigned)n_scan) {
    scan_la_block<C, DK, true>(sa, maps, blockIdx.x, sm, ready);
    return;
  }
  // ---- prep CTA: three warpgroups, each its own slice and 128 columns ----
  using PS = PrepTmemSmem<C>;
  const int wg = threadIdx.x >> 7;
  // the address slot: the first word at kMisc of warpgroup 0's slice, which
  // the unit leaves to its caller
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + PS::kMisc);
  constexpr uint32_t kCols = 512;
  unsigned char *wsm = sm + wg * PS::kSlice;
  if (threadIdx.x < 32) tmem_alloc(smem_addr(tslot), kCols);
  if ((threadIdx.x & 127) == 0 && wg < kPrepGroups) prep_tmem_init_barriers<C>(wsm);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tslot;
  if (wg < kPrepGroups) {
    const int groups = (gridDim.x - n_scan) * kPrepGroups;
    const int units = pa.n_slots * pa.H;
    PrepPhases ph;  // the slice's barriers stay initialised across units
    for (int u = unit0 + (blockIdx.x - n_scan) * kPrepGroups + wg; u < units; u += groups)
      prep_tmem_unit<C, DK>(pa, maps, u / pa.H, u % pa.H, wsm, tmem + 128u * wg,
                            threadIdx.x & 127, 1 + wg, ready, ph);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (threadIdx.x < 32) tmem_dealloc(tmem, kCols);
}

template <int C, int DK>
cudaError_t launch_one(const PrepArgs &pa, const ScanArgs &sa, const ScanMaps &maps,
                       int *ready, int head_slots, cudaStream_t stream) {
  using SM = LockSmem<C, DK>;
  auto kern = gdn_lockstep_kernel<C, DK>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (err != cudaSuccess) return err;
  int dev = 0, n_sm = 0, per_sm = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, SM::kBytes)) !=
      cudaSuccess)
    return err;
  const long n_scan = (long)sa.seq.n_seqs * sa.HV * (sa.dv / kScanTcSlice);
  const long resident = (long)n_sm * per_sm;
  if (per_sm < 1 || n_scan + 1 > resident) return cudaErrorCooperativeLaunchTooLarge;
  // The head start: the split prep kernel over the first head_slots slots.
  // The cooperative launch's prep warpgroups ((n_sm - n_scan) x 3) must
  // finish the other units while the scan walks its chain; measured on this
  // GPU, one chunk step of the scan takes about kStepPerUnit of a prep unit
  // at three per SM (1.2 against 24 us).  The head start runs in whole waves
  // of the split prep (n_sm x 4 CTAs at once), so its units are rounded up to
  // a wave and its slots down (a few more units in the next wave would cost a
  // whole unit's time).  At 32k tokens (H = 16, 96 scan blocks) this covers
  // 0.52 of the slots, at 4096 tokens 0.59 of them; swept from 0.025 to 0.1,
  // 0.05 is the best from 8192 tokens up.
  if (head_slots < 0) {
    constexpr double kStepPerUnit = 0.05;
    constexpr long kPrepPerSm = 4;  // split prep CTAs per SM
    const long units = (long)pa.n_slots * pa.H;
    const long chain = pa.seq.cu ? ((long)pa.seq.Ttot + (long)C * pa.seq.n_seqs - 1) / ((long)C * pa.seq.n_seqs)
                                 : ((long)pa.seq.T + C - 1) / C;
    const long groups = (resident - n_scan) * kPrepGroups;
    const long need = units - (long)((double)groups * (double)chain * kStepPerUnit);
    const long wave = (long)n_sm * kPrepPerSm;
    const long head_units = need <= 0 ? 0 : (need + wave - 1) / wave * wave;
    head_slots = (int)(head_units / pa.H);
  }
  head_slots = head_slots > pa.n_slots ? pa.n_slots : head_slots;
  if (head_slots > 0 &&
      (err = launch_prep_tmem(pa, maps, C, DK, stream, head_slots, ready)) != cudaSuccess)
    return err;
  int n_scan_i = (int)n_scan;
  int unit0 = head_slots * pa.H;
  PrepArgs pa_ = pa;
  ScanArgs sa_ = sa;
  ScanMaps maps_ = maps;
  void *args[] = {&pa_, &sa_, &maps_, &n_scan_i, &ready, &unit0};
  return cudaLaunchCooperativeKernel((const void *)kern, dim3((unsigned)resident), dim3(kThreads),
                                     args, SM::kBytes, stream);
}

}  // namespace

cudaError_t launch_lockstep(const PrepArgs &pa, const ScanArgs &sa, const ScanMaps &maps,
                            int *ready, int head_slots, int chunk, int dk, cudaStream_t stream) {
  if (chunk == 64 && dk == 128) return launch_one<64, 128>(pa, sa, maps, ready, head_slots, stream);
  if (chunk == 64 && dk == 64) return launch_one<64, 64>(pa, sa, maps, ready, head_slots, stream);
  if (chunk == 32 && dk == 128) return launch_one<32, 128>(pa, sa, maps, ready, head_slots, stream);
  if (chunk == 32 && dk == 64) return launch_one<32, 64>(pa, sa, maps, ready, head_slots, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
