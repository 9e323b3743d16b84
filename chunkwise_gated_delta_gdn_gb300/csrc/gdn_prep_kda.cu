// gdn_prep_kda.cu -- the chunk-prep kernel of the bf16 per-key-gate (KDA)
// path at chunk 32 (other chunk sizes run gdn_prep_tc.cu; both write the same
// outputs for the scan kernel gdn_scan_tc.cu).
//
// One CTA (128 threads) per (chunk slot, value head), five per SM at dk = 128
// (45 KB of shared memory, 80 registers and 64 tensor-memory columns each),
// four at dk = 64.  The chunk's key,
// query and gate tiles arrive by TMA.  The gates are summed along the chunk
// per key channel, b_r = sum_{j <= r} g_j (log2 units here), and every
// exponential of the chunk is taken against one reference row m = 16:
//   E_rc = 2^(b_rc - b_mc),   E_rc^-1 = 2^(b_mc - b_rc)
// With them, in one pass over the tile (ROCm/rocm-libraries PR #11223,
// "Summary": the per-channel decays enter the products as factors of their
// operands, "Correctness": no exponent is formed that could overflow):
//   K~ = K E,  Q~ = Q E,  K^ = K E^-1          (operands of A and Aqk)
//   Kg = K E 2^b_m,  Qg = scale Q E 2^b_m       (= K 2^b, the scan's gated image)
//   Kt = K E^-1 2^(b_last - b_m)                (= K 2^(b_last - b), for P1)
// so that
//   A   = strict-lower(beta_r (K~ K^^T)_rs)     Aqk = lower(scale (Q~ K^^T)_rs)
// is one tensor-core product [K~; Q~] K^^T per 64-channel panel, in split
// bf16: each factored operand as hi + lo bf16 planes (16 significant bits and
// the fp32 exponent range), hi hi + lo hi + hi lo accumulated in fp32 in
// tensor memory.  While every |b_rc - b_mc| <= 100 (log2 units) every factor
// and its low part stay normal fp32 / bf16 numbers; a chunk whose gates reach
// further (sums of 16 gates below about -69 in natural-log units) forms each
// pairwise decay directly instead, as the exact reading requires.
// Then, as in gdn_prep_tc.cu:
//   T    = (I + A)^-1   (16 x 16 diagonal blocks by forward substitution, then
//          the block row)
//   P1   = Kt^T T,  AqkT = Aqk T   (tcgen05, fp16 operands, fp32 accumulation)
// written, rounded once to fp16, as the 10 KB image [P1; AqkT] (K-major,
// 64-byte swizzle, 160 rows of 32 elements) with one bulk copy; the gated
// image [Kg; Qg] (per 64-channel panel 2C rows: the keys, then the queries;
// rows past the tokens zero) and e^{b_last} per key channel go straight to
// global memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kC = 32;     // chunk
constexpr int kNT = 128;   // threads
constexpr int kRef = 16;   // reference row of the factored exponentials
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kWide = 100.f;  // largest |b_r - b_ref| (log2 units) for the factored form
// the gated [Kg; Qg] image: per 64-channel panel, the C key rows then the C
// query rows (128-byte rows, 128-byte swizzle)
constexpr int kKqPanel = 2 * kC * 128;

__device__ __forceinline__ float ex2k(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int DK>
struct KdaSmem {
  static constexpr int NP = DK / 64;  // 64-channel panels
  // dk = 128 builds the factored planes per 32-channel half panel (64-byte
  // swizzle, 12 KB) and puts the solve's fp32 T and scratch, and Kt, over the
  // gate tile once it is dead, so that five CTAs share an SM; dk = 64 fits
  // four with whole-panel planes
  static constexpr bool HALF = DK == 128;
  static constexpr int NH = HALF ? 2 * NP : NP;  // plane products per unit
  // TMA tiles: K and Q bf16 (C rows x 128 bytes per panel, 128-byte swizzle),
  // gates fp32 (C rows x 256 bytes per panel), summed in place
  static constexpr int kK = 0;
  static constexpr int kQ = kK + NP * kC * 128;
  static constexpr int kG = kQ + NP * kC * 128;
  // the factored operands of one panel (K-major): [K~; Q~] hi and lo (64 rows
  // each), K^ hi and lo (32 rows each); 128-byte rows (whole panel) or 64-byte
  // rows (half panel)
  static constexpr int kPl = kG + NP * kC * 256;
  static constexpr int ROWB = HALF ? 64 : 128;
  static constexpr int PL_AH = 0, PL_AL = 64 * ROWB, PL_BH = 128 * ROWB, PL_BL = 160 * ROWB;
  static constexpr int PLANES = 192 * ROWB;
  // Kt as fp16 token rows, two 64-channel panels (P1's M = 128 reads both).
  // dk = 128: over the gate tile's second panel, written once the tile is
  // dead (each thread holds its share in registers from the plane passes
  // until then), so that five CTAs share an SM; dk = 64: after the planes
  static constexpr int kKt = HALF ? kG + kC * 256 : kPl + PLANES;
  static constexpr int kBeta = HALF ? kPl + PLANES : kKt + 2 * kC * 128;
  static constexpr int kBar = kBeta + kC * 4;  // TMA tiles, products
  static constexpr int kTslot = kBar + 16;
  static constexpr int kAbort = kTslot + 4;
  static constexpr int kMeta = kAbort + 4;
  // 1 KB of alignment slack, except at dk = 128, where the kernel checks
  // that the dynamic shared memory it received is already 1 KB aligned
  static constexpr int kSlack = HALF ? 0 : 1024;
  static constexpr int kBytes = kMeta + 16 + kSlack;
  static constexpr int kPerSm = HALF ? 5 : 4;  // CTAs per SM
  // once the A / Aqk products have read the planes, their region holds fp32 A
  // (and, on the strong-decay path, fp32 Aqk), then the fp16 T image (B
  // operand), then the output image; fp32 T and the solve's scratch lie over
  // the dead gate tile (half panels) or in the plane region after A; the fp16
  // Aqk operand (A of a M = 128 product: 16 KB from its base) lies over the
  // dead K / Q tiles
  static constexpr int LDC = kC + 4;
  static constexpr int ARR = kC * LDC * 4;  // one C x C fp32 array
  static constexpr int kAs = kPl;
  static constexpr int kTs = HALF ? kG : kAs + ARR;
  static constexpr int kRs = kTs + ARR;
  static constexpr int kAqkF = HALF ? kAs + ARR : kRs + 16 * LDC * 4;
  static constexpr int kTimg = HALF ? kPl : kPl + 16384;
  static constexpr int kImg = kPl;
  static constexpr int kAqkOp = kK;
  static_assert(kAqkF + ARR <= kPl + PLANES, "fp32 A and Aqk inside the plane region");
  static_assert(!HALF || kRs + 16 * LDC * 4 <= kKt, "T and scratch below Kt in the dead gate tile");
  static_assert(!HALF || kKt + 2 * kC * 128 <= kPl, "Kt inside the dead gate tile");
  static_assert(HALF || kAqkF + ARR <= kTimg, "fp32 arrays below the T image");
  static_assert(kTimg + kC * 128 <= kPl + PLANES, "T image inside the planes region");
  static_assert(kPrepImage32Bytes <= PLANES, "output image inside the planes region");
  static_assert(kPl - kK >= 16384, "the Aqk operand's 128-row span over the dead tiles");
  static_assert(kBar % 8 == 0 && kPl % 1024 == 0 && kKt % 1024 == 0, "alignment");
  // 228 KB of shared memory per SM, 1 KB of it reserved per CTA
  static_assert(kPerSm * (kBytes + 1024) <= 233472, "CTAs per SM");
};

// At most 80 registers a thread (the bound for six CTAs; shared memory allows
// five): a prep CTA then also fits beside a scan CTA of gdn_scan_tc.cu
// (55.3K + 10.2K of the SM's 64K registers), where batches in flight run one
// batch's prep on the SMs another batch's scan holds.
template <int DK>
__global__ void __launch_bounds__(kNT, 6)
gdn_prep_kda_kernel(const PrepArgs a, const __grid_constant__ ScanMaps maps) {
  using SM = KdaSmem<DK>;
  constexpr int NP = SM::NP, C = kC, LDC = SM::LDC;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  if (sm - smem_raw > SM::kSlack) {  // dynamic shared memory not aligned as needed
    if (threadIdx.x == 0) atomicOr(a.flags, kFlagLaunchConfig);
    return;
  }
  float *Bs = reinterpret_cast<float *>(sm + SM::kBeta);
  int *meta = reinterpret_cast<int *>(sm + SM::kMeta);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + SM::kTslot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SM::kAbort);
  const uint32_t bar_tma = smem_addr(sm + SM::kBar), bar_mma = bar_tma + 8;

  const int slot = blockIdx.x, hv = blockIdx.y;
  const int hq = hv / (a.HV / a.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- slot -> (sequence, chunk) ----
  if (tid == 0) {
    int lo = 0, hi = a.seq.n_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (slot_base<C>(a.seq, mid) <= slot) lo = mid; else hi = mid - 1;
    }
    int start, end;
    int valid = seq_ok(a.seq, lo, start, end) ? 1 : 0;
    const long c = (long)slot - slot_base<C>(a.seq, lo);
    const long t0 = (long)start + c * C;
    if (c < 0 || t0 >= end) valid = 0;
    meta[0] = valid ? (int)t0 : 0;
    meta[1] = valid ? (int)min((long)C, (long)end - t0) : 0;
    meta[2] = valid;
  }
  __syncthreads();
  if (!meta[2]) return;  // unused slot: the scan never reads it
  const int t0 = meta[0], L = meta[1];

  // ---- set-up, tiles by TMA ----
  // A / Aqk at 0, then (once they are read out) P1 at 0 and Aqk T at 32: 64
  // columns, so that five CTAs fit the SM's 512
  constexpr uint32_t kTmemCols = 64;
  if (warp == 0) tmem_alloc(smem_addr(tslot), kTmemCols);
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(bar_tma, NP * C * (128 + 128 + 256));
#pragma unroll
    for (int p = 0; p < NP; p++) {
      tma_load_3d(smem_addr(sm + SM::kK + p * C * 128), &maps.k, p * 64, hq, t0, bar_tma);
      tma_load_3d(smem_addr(sm + SM::kQ + p * C * 128), &maps.q, p * 64, hq, t0, bar_tma);
      tma_load_3d(smem_addr(sm + SM::kG + p * C * 256), &maps.g, p * 64, hv, t0, bar_tma);
    }
  }
  if (tid < C) Bs[tid] = tid < L ? __ldg(a.beta + (long)(t0 + tid) * a.HV + hv) : 0.f;
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tslot;
  mbar_wait(bar_tma, 0, abort_flag);
  // rows past the chunk's tokens (the next sequence's, in packed input) -> 0
  if (L < C) {
    for (int idx = tid; idx < NP * (C - L) * 8; idx += kNT) {
      const int p = idx / ((C - L) * 8), r = L + (idx / 8) % (C - L), ch = idx % 8;
      *reinterpret_cast<uint4 *>(sm + SM::kK + p * C * 128 + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(sm + SM::kQ + p * C * 128 + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(sm + SM::kG + p * C * 256 + r * 256 + ch * 32) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(sm + SM::kG + p * C * 256 + r * 256 + ch * 32 + 16) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
  }

  // ---- cumulative gates per key channel (log2 units), in place ----
  bool positive = false, wide = false;
  if (tid < DK) {
    float *gcol = reinterpret_cast<float *>(sm + SM::kG + (tid >> 6) * C * 256) + (tid & 63);
    float run = 0.f, bmin = 0.f, bmax = 0.f, bref = 0.f;
#pragma unroll 8
    for (int r = 0; r < C; r++) {
      const float g = gcol[r * 64];
      positive |= g > 0.f;
      run = fmaf(g, kLog2e, run);
      gcol[r * 64] = run;
      bmin = fminf(bmin, run);
      bmax = fmaxf(bmax, run);
      if (r == kRef) bref = run;
    }
    wide = fmaxf(bmax - bref, bref - bmin) > kWide;
  }
  if (__syncthreads_or(positive) && tid == 0) atomicOr(a.flags, kFlagPositiveGate);
  wide = __syncthreads_or(wide);

  // ---- one pass over the tile per 64-channel panel (dk = 64) or 32-channel
  //      half panel (dk = 128): factored planes (and their product), the
  //      gated image, Kt, the decays ----
  // dk = 128: this thread's Kt values (half panel hp, row 4 rg + i, channel
  // pair pp), held until the gate tile is dead
  uint32_t ktr[SM::HALF ? SM::NH : 1][4];
  if constexpr (SM::HALF) {
    // 32-channel half panels hp: 16 channel pairs x 8 groups of 4 rows; the
    // planes in the 64-byte swizzle, one K = 32 product per half panel
    const int pp = tid & 15, rg = tid >> 4;
    unsigned char *kqi = a.kq_images + ((size_t)slot * a.HV + hv) * kq_image_bytes(DK);
    const uint32_t sPl = smem_addr(sm + SM::kPl);
#pragma unroll
    for (int hp = 0; hp < SM::NH; hp++) {
      const int p = hp >> 1, col = 32 * (hp & 1) + 2 * pp;  // first channel of the pair in the panel
      const int kc = col & 31;                                 // and in the half panel
      if (!wide && hp > 0) {  // the previous half panel's products have read the planes
        mbar_wait(bar_mma, (hp - 1) & 1, abort_flag);
        fence_after_sync();
      }
      const float *gp = reinterpret_cast<const float *>(sm + SM::kG + p * C * 256);
      const float2 bm = *reinterpret_cast<const float2 *>(gp + kRef * 64 + col);
      const float2 bl = *reinterpret_cast<const float2 *>(gp + (C - 1) * 64 + col);
      const float ebm0 = ex2k(bm.x), ebm1 = ex2k(bm.y);
      const float elt0 = ex2k(bl.x - bm.x), elt1 = ex2k(bl.y - bm.y);
      if (rg == 0)
        *reinterpret_cast<float2 *>(a.decays + ((size_t)slot * a.HV + hv) * DK + p * 64 + col) =
            make_float2(ex2k(bl.x), ex2k(bl.y));
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int r = 4 * rg + i;
        // element (r, col) of a 64-channel K-major row in the 128-byte swizzle,
        // and (r, kc) of a 32-channel row in the 64-byte swizzle
        const uint32_t off = r * 128 + ((((col >> 3) ^ (r & 7)) << 4) | ((col & 7) * 2));
        const float2 b = *reinterpret_cast<const float2 *>(gp + r * 64 + col);
        const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm + SM::kK + p * C * 128 + off));
        const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm + SM::kQ + p * C * 128 + off));
        float kg0, kg1, qg0, qg1, kt0, kt1;
        if (!wide) {
          const float e0 = ex2k(b.x - bm.x), e1 = ex2k(b.y - bm.y);
          const float i0 = ex2k(bm.x - b.x), i1 = ex2k(bm.y - b.y);
          uint32_t h, l;
          split2(kf.x * e0, kf.y * e1, h, l);
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_AH + kmajor64_off(r, kc)) = h;
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_AL + kmajor64_off(r, kc)) = l;
          split2(qf.x * e0, qf.y * e1, h, l);
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_AH + kmajor64_off(32 + r, kc)) = h;
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_AL + kmajor64_off(32 + r, kc)) = l;
          split2(kf.x * i0, kf.y * i1, h, l);
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_BH + kmajor64_off(r, kc)) = h;
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_BL + kmajor64_off(r, kc)) = l;
          kg0 = kf.x * e0 * ebm0; kg1 = kf.y * e1 * ebm1;
          qg0 = a.scale * qf.x * e0 * ebm0; qg1 = a.scale * qf.y * e1 * ebm1;
          kt0 = kf.x * i0 * elt0; kt1 = kf.y * i1 * elt1;
        } else {
          const float eb0 = ex2k(b.x), eb1 = ex2k(b.y);
          kg0 = kf.x * eb0; kg1 = kf.y * eb1;
          qg0 = a.scale * qf.x * eb0; qg1 = a.scale * qf.y * eb1;
          kt0 = kf.x * ex2k(bl.x - b.x); kt1 = kf.y * ex2k(bl.y - b.y);
        }
        const __half2 kg = __floats2half2_rn(kg0, kg1), qg = __floats2half2_rn(qg0, qg1);
        *reinterpret_cast<__half2 *>(kqi + p * kKqPanel + off) = kg;
        *reinterpret_cast<__half2 *>(kqi + p * kKqPanel + kC * 128 + off) = qg;
        const __half2 kt = __floats2half2_rn(kt0, kt1);
        ktr[hp][i] = *reinterpret_cast<const uint32_t *>(&kt);
      }
      if (!wide) {
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (tid == 0) {
          // [K~; Q~] K^^T over the half panel's 32 channels (M = 128: rows 64..
          // are not read back), hi hi + lo hi + hi lo
          constexpr uint32_t id = idesc_bf16(128, C, 0, 0);
#pragma unroll
          for (int k0 = 0; k0 < 32; k0 += 16) {
            const uint64_t ah = make_desc_sw64(sPl + SM::PL_AH + k0 * 2, 512);
            const uint64_t al = make_desc_sw64(sPl + SM::PL_AL + k0 * 2, 512);
            const uint64_t bh = make_desc_sw64(sPl + SM::PL_BH + k0 * 2, 512);
            const uint64_t bo = make_desc_sw64(sPl + SM::PL_BL + k0 * 2, 512);
            mma_f16(tmem, ah, bh, id, (hp > 0 || k0 > 0) ? 1u : 0u);
            mma_f16(tmem, al, bh, id, 1u);
            mma_f16(tmem, ah, bo, id, 1u);
          }
          mma_commit(bar_mma);
        }
      }
    }
  } else
  {
    const int pp = tid & 31, rg = tid >> 5;  // channel pair, group of 8 rows
    const int col = 2 * pp;                  // first channel of the pair in the panel
    unsigned char *kqi = a.kq_images + ((size_t)slot * a.HV + hv) * kq_image_bytes(DK);
    const uint32_t sPl = smem_addr(sm + SM::kPl);
#pragma unroll 1
    for (int p = 0; p < NP; p++) {
      if (!wide && p > 0) {  // the previous panel's products have read the planes
        mbar_wait(bar_mma, (p - 1) & 1, abort_flag);
        fence_after_sync();
      }
      const float *gp = reinterpret_cast<const float *>(sm + SM::kG + p * C * 256);
      const float2 bm = *reinterpret_cast<const float2 *>(gp + kRef * 64 + col);
      const float2 bl = *reinterpret_cast<const float2 *>(gp + (C - 1) * 64 + col);
      const float ebm0 = ex2k(bm.x), ebm1 = ex2k(bm.y);
      const float elt0 = ex2k(bl.x - bm.x), elt1 = ex2k(bl.y - bm.y);
      if (rg == 0)
        *reinterpret_cast<float2 *>(a.decays + ((size_t)slot * a.HV + hv) * DK + p * 64 + col) =
            make_float2(ex2k(bl.x), ex2k(bl.y));
#pragma unroll 2
      for (int i = 0; i < 8; i++) {
        const int r = 8 * rg + i;
        // element (r, col) of a 64-channel K-major row in the 128-byte swizzle
        const uint32_t off = r * 128 + ((((col >> 3) ^ (r & 7)) << 4) | ((col & 7) * 2));
        const float2 b = *reinterpret_cast<const float2 *>(gp + r * 64 + col);
        const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm + SM::kK + p * C * 128 + off));
        const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm + SM::kQ + p * C * 128 + off));
        float kg0, kg1, qg0, qg1, kt0, kt1;
        if (!wide) {
          const float e0 = ex2k(b.x - bm.x), e1 = ex2k(b.y - bm.y);
          const float i0 = ex2k(bm.x - b.x), i1 = ex2k(bm.y - b.y);
          uint32_t h, l;
          split2(kf.x * e0, kf.y * e1, h, l);
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_AH + off) = h;
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_AL + off) = l;
          split2(qf.x * e0, qf.y * e1, h, l);
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_AH + 32 * 128 + off) = h;
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_AL + 32 * 128 + off) = l;
          split2(kf.x * i0, kf.y * i1, h, l);
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_BH + off) = h;
          *reinterpret_cast<uint32_t *>(sm + SM::kPl + SM::PL_BL + off) = l;
          kg0 = kf.x * e0 * ebm0; kg1 = kf.y * e1 * ebm1;
          qg0 = a.scale * qf.x * e0 * ebm0; qg1 = a.scale * qf.y * e1 * ebm1;
          kt0 = kf.x * i0 * elt0; kt1 = kf.y * i1 * elt1;
        } else {
          const float eb0 = ex2k(b.x), eb1 = ex2k(b.y);
          kg0 = kf.x * eb0; kg1 = kf.y * eb1;
          qg0 = a.scale * qf.x * eb0; qg1 = a.scale * qf.y * eb1;
          kt0 = kf.x * ex2k(bl.x - b.x); kt1 = kf.y * ex2k(bl.y - b.y);
        }
        const __half2 kg = __floats2half2_rn(kg0, kg1), qg = __floats2half2_rn(qg0, qg1);
        *reinterpret_cast<__half2 *>(kqi + p * kKqPanel + off) = kg;
        *reinterpret_cast<__half2 *>(kqi + p * kKqPanel + kC * 128 + off) = qg;
        *reinterpret_cast<__half2 *>(sm + SM::kKt + p * C * 128 + off) = __floats2half2_rn(kt0, kt1);
      }
      if (!wide) {
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (tid == 0) {
          // [K~; Q~] K^^T over the panel's 64 channels (M = 128: rows 64.. are
          // not read back), hi hi + lo hi + hi lo
          constexpr uint32_t id = idesc_bf16(128, C, 0, 0);
#pragma unroll
          for (int k0 = 0; k0 < 64; k0 += 16) {
            const uint64_t ah = make_desc(sPl + SM::PL_AH + k0 * 2, 16, 1024);
            const uint64_t al = make_desc(sPl + SM::PL_AL + k0 * 2, 16, 1024);
            const uint64_t bh = make_desc(sPl + SM::PL_BH + k0 * 2, 16, 1024);
            const uint64_t bo = make_desc(sPl + SM::PL_BL + k0 * 2, 16, 1024);
            mma_f16(tmem, ah, bh, id, (p > 0 || k0 > 0) ? 1u : 0u);
            mma_f16(tmem, al, bh, id, 1u);
            mma_f16(tmem, ah, bo, id, 1u);
          }
          mma_commit(bar_mma);
        }
      }
    }
  }

  float *As = reinterpret_cast<float *>(sm + SM::kAs);
  float *Ts = reinterpret_cast<float *>(sm + SM::kTs);
  float *Rs = reinterpret_cast<float *>(sm + SM::kRs);
  unsigned char *opAqk = sm + SM::kAqkOp;
  if (!wide) {
    // ---- A (lanes 0..31) and Aqk (lanes 32..63) from tensor memory ----
    mbar_wait(bar_mma, (SM::NH - 1) & 1, abort_flag);
    fence_after_sync();
    if (warp < 2) {
      uint32_t v[32];
      tmem_ld32_nowait(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
      tmem_wait_ld();
      const int r = lane;
      if (warp == 0) {
        const float br = Bs[r];
#pragma unroll
        for (int s = 0; s < C; s++) As[r * LDC + s] = s < r ? br * __uint_as_float(v[s]) : 0.f;
      } else {
#pragma unroll
        for (int ch = 0; ch < 8; ch++) {
          uint4 pk = make_uint4(0, 0, 0, 0);
          if (ch < C / 8) {
            __half2 *h = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const int s = ch * 8 + 2 * i;
              h[i] = __floats2half2_rn(s <= r ? a.scale * __uint_as_float(v[s]) : 0.f,
                                       s + 1 <= r ? a.scale * __uint_as_float(v[s + 1]) : 0.f);
            }
          }
          *reinterpret_cast<uint4 *>(opAqk + kmajor_off(r, ch * 8, 128)) = pk;
        }
      }
    }
  } else {
    // ---- strong decays: every pairwise decay formed directly ----
    float *AqkF = reinterpret_cast<float *>(sm + SM::kAqkF);
    const float *G = reinterpret_cast<const float *>(sm + SM::kG);
    auto tile = [&](int base, int r, int c) {  // element (r, c) of a bf16 K / Q tile
      const int p = c >> 6, cc = c & 63;
      const uint32_t off = p * C * 128 + r * 128 + ((((cc >> 3) ^ (r & 7)) << 4) | ((cc & 7) * 2));
      return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + base + off));
    };
    constexpr int NPAIR = C * (C + 1) / 2;
    for (int pr = warp; pr < NPAIR; pr += kNT / 32) {
      int r = (int)((sqrtf(8.f * pr + 1.f) - 1.f) * 0.5f);
      while ((r + 1) * (r + 2) / 2 <= pr) r++;
      while (r * (r + 1) / 2 > pr) r--;
      const int s = pr - r * (r + 1) / 2;
      float kk = 0.f, qk = 0.f;
      for (int c = lane; c < DK; c += 32) {
        const float *gc = G + (c >> 6) * C * 64 + (c & 63);
        const float ks = tile(SM::kK, s, c) * ex2k(gc[r * 64] - gc[s * 64]);
        kk = fmaf(tile(SM::kK, r, c), ks, kk);
        qk = fmaf(tile(SM::kQ, r, c), ks, qk);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        kk += __shfl_xor_sync(0xffffffffu, kk, off);
        qk += __shfl_xor_sync(0xffffffffu, qk, off);
      }
      if (lane == 0) {
        As[r * LDC + s] = s < r ? Bs[r] * kk : 0.f;
        AqkF[r * LDC + s] = a.scale * qk;
      }
    }
    __syncthreads();  // every reader of the tiles is done: the operand goes over them
    for (int idx = tid; idx < C * 8; idx += kNT) {
      const int r = idx >> 3, ch = idx & 7;
      uint4 pk = make_uint4(0, 0, 0, 0);
      if (ch < C / 8) {
        __half2 *h = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const int s = ch * 8 + 2 * i;
          h[i] = __floats2half2_rn(s <= r ? AqkF[r * LDC + s] : 0.f, s + 1 <= r ? AqkF[r * LDC + s + 1] : 0.f);
        }
      }
      *reinterpret_cast<uint4 *>(opAqk + kmajor_off(r, ch * 8, 128)) = pk;
    }
    for (int idx = tid; idx < C * C; idx += kNT) {
      const int r = idx / C, s = idx % C;
      if (s >= r) As[r * LDC + s] = 0.f;
    }
  }
  __syncthreads();
  if constexpr (SM::HALF) {
    // every reader of the gate tile is done: Kt over its second panel
    const int pp = tid & 15, rg = tid >> 4;
#pragma unroll
    for (int hp = 0; hp < SM::NH; hp++) {
      const int p = hp >> 1, col = 32 * (hp & 1) + 2 * pp;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int r = 4 * rg + i;
        const uint32_t off = r * 128 + ((((col >> 3) ^ (r & 7)) << 4) | ((col & 7) * 2));
        *reinterpret_cast<uint32_t *>(sm + SM::kKt + p * C * 128 + off) = ktr[hp][i];
      }
    }
    fence_proxy_async();
  }

  // ---- T = (I + A)^-1 ----
  constexpr int NB = C / 16;
  if (tid < NB * 16) {
    // diagonal block I, column j: forward substitution
    const int I = tid / 16, j = tid % 16, o = 16 * I;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; r++) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
    for (int s = 0; s < 16; s++) {
      const float xs = x[s];
#pragma unroll
      for (int r = s + 1; r < 16; r++) x[r] -= As[(o + r) * LDC + o + s] * xs;
    }
#pragma unroll
    for (int r = 0; r < 16; r++) Ts[(o + r) * LDC + o + j] = x[r];
  }
  for (int idx = tid; idx < 16 * 16; idx += kNT) Ts[(idx / 16) * LDC + 16 + idx % 16] = 0.f;  // upper block
  __syncthreads();
  // block row 1:  R = A[1, 0] T[0, 0],  T[1, 0] = -T[1, 1] R
  for (int idx = tid; idx < 16 * 16; idx += kNT) {
    const int m = idx / 16, j = idx % 16;
    float acc = 0.f;
#pragma unroll
    for (int s = 0; s < 16; s++) acc = fmaf(As[(16 + m) * LDC + s], Ts[s * LDC + j], acc);
    Rs[m * LDC + j] = acc;
  }
  __syncthreads();
  for (int idx = tid; idx < 16 * 16; idx += kNT) {
    const int m = idx / 16, j = idx % 16;
    float acc = 0.f;
    for (int p = 0; p <= m; p++) acc = fmaf(Ts[(16 + m) * LDC + 16 + p], Rs[p * LDC + j], acc);
    Ts[(16 + m) * LDC + j] = -acc;
  }
  __syncthreads();

  // ---- T as the B operand of the image products: row j = T[.][j], 64
  //      columns (zero beyond C) ----
  unsigned char *opT = sm + SM::kTimg;
  for (int idx = tid; idx < C * 8; idx += kNT) {
    const int j = idx >> 3, ch = idx & 7;
    uint4 pk = make_uint4(0, 0, 0, 0);
    if (ch < C / 8) {
      __half2 *h = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int k = ch * 8 + 2 * i;
        h[i] = __floats2half2_rn(Ts[k * LDC + j], Ts[(k + 1) * LDC + j]);
      }
    }
    *reinterpret_cast<uint4 *>(opT + kmajor_off(j, ch * 8, C)) = pk;
  }
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  // ---- P1 = Kt^T T (M = dk rows, read MN-major; N = K = C) and Aqk T ----
  if (tid == 0) {
    const uint32_t sKt = smem_addr(sm + SM::kKt), sT = smem_addr(opT), sAqk = smem_addr(opAqk);
    constexpr uint32_t idP = idesc_f16(128, C, 1, 0);
    constexpr uint32_t idQ = idesc_f16(128, C, 0, 0);
#pragma unroll
    for (int k0 = 0; k0 < C; k0 += 16) {
      const uint64_t bd = make_desc(sT + k0 * 2, 16, 1024);
      mma_f16(tmem, make_desc(sKt + k0 * 128, C * 128, 1024), bd, idP, k0 > 0 ? 1u : 0u);
      mma_f16(tmem + 32, make_desc(sAqk + k0 * 2, 16, 1024), bd, idQ, k0 > 0 ? 1u : 0u);
    }
    mma_commit(bar_mma);
  }
  mbar_wait(bar_mma, (wide ? 0 : SM::NH) & 1, abort_flag);
  fence_after_sync();

  // ---- the image [P1; AqkT], 32 columns per row in the 64-byte swizzle:
  //      row t of P1 (zero for t >= dk), rows 128 + r of AqkT ----
  unsigned char *img = sm + SM::kImg;
  {
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    auto put_row = [&](int row, uint32_t taddr, bool have) {
      uint32_t v[32];
      if (have) {
        tmem_ld32_nowait(taddr, v);
        tmem_wait_ld();
      }
#pragma unroll
      for (int ch = 0; ch < C / 8; ch++) {
        uint4 pk = make_uint4(0, 0, 0, 0);
        if (have) {
          __half2 *hh = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
          for (int i = 0; i < 4; i++)
            hh[i] = __floats2half2_rn(__uint_as_float(v[ch * 8 + 2 * i]), __uint_as_float(v[ch * 8 + 2 * i + 1]));
        }
        *reinterpret_cast<uint4 *>(img + kmajor64_off(row, ch * 8)) = pk;
      }
    };
    // tensor-memory loads are warp-wide: every lane of a warp loads
    put_row(tid, tmem + lane_base, warp * 32 < DK);
    if (warp == 0) put_row(128 + tid, tmem + lane_base + 32, true);
  }
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  // ---- image -> workspace, one bulk copy ----
  if (tid == 0) {
    unsigned char *dst = reinterpret_cast<unsigned char *>(a.tiles) + ((size_t)slot * a.HV + hv) * kPrepImageBytes;
    bulk_s2g(dst, smem_addr(img), kPrepImage32Bytes);
    bulk_commit();
    bulk_wait_read_all();
    if (*abort_flag) atomicOr(a.flags, kFlagTimeout);
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int DK>
cudaError_t launch_one(const PrepArgs &a, const ScanMaps &maps, cudaStream_t stream) {
  using SM = KdaSmem<DK>;
  auto kern = gdn_prep_kda_kernel<DK>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (err != cudaSuccess) return err;
  kern<<<dim3(a.n_slots, a.HV), kNT, SM::kBytes, stream>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_kda(const PrepArgs &a, const ScanMaps &maps, int dk, cudaStream_t stream) {
  if (dk == 128) return launch_one<128>(a, maps, stream);
  if (dk == 64) return launch_one<64>(a, maps, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
