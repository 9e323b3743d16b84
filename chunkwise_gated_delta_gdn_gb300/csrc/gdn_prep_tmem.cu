// gdn_prep_tmem.cu -- chunk-prep kernel of the bf16 scalar-gate (GDN) path on
// the 5th-generation tensor cores.
//
// One CTA (128 threads) per (chunk slot, value head).  It produces the same
// 24 KB fp16 operand image as the generic bf16 prep (rows 0..127 = P1 = Kt^T T,
// rows 128..191 = Aqk T; K-major, 128-byte swizzle), through three tensor-core
// products with accumulators in tensor memory:
//   G  = [K; Q] K^T          M = 128 (keys then queries), N = C, K = dk
//   P1 = K^T (D T)           A = the key tile read MN-major (M = dk, K = C),
//                            D = diag(exp(b_last - b_s))
//   AqkT = Aqk T             K = C
// Between them, in fp32: A = strict-lower(beta_r G_rs exp(b_r - b_s)) and
// Aqk = lower(scale P_rs exp(b_r - b_s)) straight from each thread's tensor-
// memory lane (pairwise decays only for s <= r, so no exponent is positive),
// and T = (I + A)^-1 by the blocked solve of ROCm/rocm-libraries PR #11223
// ("Levers" 3): 16 x 16 diagonal blocks by forward substitution, then block
// rows by products against the solved blocks, in place.  Keys and queries
// arrive by TMA (bf16, 128-byte swizzle) and are converted to fp16 in place;
// the fp16 operands of the three products (11-bit mantissa) and of the image
// are the only roundings.
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

constexpr int kThreads = 128;

template <int C, int DK>
struct PrepTmemSmem {
  static constexpr int LDC = C + 4;              // fp32 row stride of A / T
  static constexpr int KQ = 2 * 128 * 128;       // [K; Q] image, always two panels
  static constexpr int kKQ = 0;                  // later: the output image
  static constexpr int kAqk = kKQ + KQ;          // Aqk, K-major, 64 rows (8 KB)
  static constexpr int kTi = kAqk + 8 * 1024;    // T, MN-major, 64 K-rows (8 KB)
  static constexpr int kDTi = kTi + 8 * 1024;    // D T, MN-major (8 KB)
  static constexpr int kA = kDTi + 8 * 1024;     // A -> T, fp32
  static constexpr int kR = kA + C * LDC * 4;    // 16 x LDC scratch
  static constexpr int kG = kR + 16 * LDC * 4;   // gates -> cumulative gates
  static constexpr int kBeta = kG + C * 4;
  static constexpr int kDec = kBeta + C * 4;     // exp(b_last - b_s)
  static constexpr int kBar = kDec + C * 4;
  static constexpr int kMisc = kBar + 16;
  static constexpr int kBytes = kMisc + 16 + 1024;
  static_assert(KQ >= kPrepImageBytes, "the output image reuses the [K; Q] region");
};

template <int C, int DK>
__global__ void __launch_bounds__(kThreads)
gdn_prep_tmem_kernel(const PrepArgs a, const __grid_constant__ ScanMaps maps) {
  using SM = PrepTmemSmem<C, DK>;
  constexpr int LDC = SM::LDC;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char *kq = sm + SM::kKQ;
  float *As = reinterpret_cast<float *>(sm + SM::kA);
  float *Rs = reinterpret_cast<float *>(sm + SM::kR);
  float *Gs = reinterpret_cast<float *>(sm + SM::kG);
  float *Bs = reinterpret_cast<float *>(sm + SM::kBeta);
  float *Ds = reinterpret_cast<float *>(sm + SM::kDec);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM::kBar);
  const uint32_t bar_tma = smem_addr(bars), bar_mma = smem_addr(bars + 1);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + SM::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SM::kMisc + 4);
  int *meta = reinterpret_cast<int *>(sm + SM::kMisc + 8);

  const int slot = blockIdx.x, hv = blockIdx.y;
  const int hq = hv / (a.HV / a.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

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
    *abort_flag = 0;
    if (valid) {
      mbar_init(bar_tma, 1);
      mbar_init(bar_mma, 1);
      mbar_fence_init();
    }
  }
  __syncthreads();
  if (!meta[2]) return;  // unused slot: the scan never reads it
  const int t0 = meta[0], L = meta[1];

  if (warp == 0) tmem_alloc(smem_addr(tslot), 128);
  // keys and queries by TMA; zero the rows no box covers (C = 32)
  if (C < 64) {
    for (int i = tid; i < SM::KQ / 16; i += kThreads) {
      const int row = (i * 16 % 16384) / 128;
      if ((row & 63) >= C) reinterpret_cast<uint4 *>(kq)[i] = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_tma, 2 * C * DK * 2);
#pragma unroll
    for (int p = 0; p < DK / 64; p++) {
      tma_load_3d(smem_addr(kq + p * 16384), &maps.k, p * 64, hq, t0, bar_tma);
      tma_load_3d(smem_addr(kq + p * 16384 + 64 * 128), &maps.q, p * 64, hq, t0, bar_tma);
    }
  }
  // gates, beta; cumulative gates (warp 0)
  bool positive = false;
  if (tid < C) {
    const float gv = tid < L ? __ldg(a.g + (long)(t0 + tid) * a.HV + hv) : 0.f;
    positive = gv > 0.f;
    Gs[tid] = gv;
    Bs[tid] = tid < L ? __ldg(a.beta + (long)(t0 + tid) * a.HV + hv) : 0.f;
  }
  if (__syncthreads_or(positive) && tid == 0) atomicOr(a.flags, kFlagPositiveGate);
  if (warp == 0) {
    float x0 = lane < C ? Gs[lane] : 0.f;
    float x1 = lane + 32 < C ? Gs[lane + 32] : 0.f;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const float y0 = __shfl_up_sync(0xffffffffu, x0, d);
      const float y1 = __shfl_up_sync(0xffffffffu, x1, d);
      if (lane >= d) { x0 += y0; x1 += y1; }
    }
    x1 += __shfl_sync(0xffffffffu, x0, 31);
    const float blast = __shfl_sync(0xffffffffu, C > 32 ? x1 : x0, (C - 1) & 31);
    if (lane < C) { Gs[lane] = x0; Ds[lane] = __expf(blast - x0); }
    if (lane + 32 < C) { Gs[lane + 32] = x1; Ds[lane + 32] = __expf(blast - x1); }
  }
  mbar_wait(bar_tma, 0, abort_flag);
  // bf16 -> fp16 in place; rows beyond the chunk's tokens -> 0
  {
    constexpr int CH = (DK / 64) * 2 * C * 8;
    for (int idx = tid; idx < CH; idx += kThreads) {
      const int p = idx / (2 * C * 8), rem = idx % (2 * C * 8);
      const int half = rem / (C * 8), r = (rem / 8) % C, chunk = rem % 8;
      uint4 *ptr = reinterpret_cast<uint4 *>(kq + p * 16384 + (half * 64 + r) * 128 + chunk * 16);
      const uint4 v = *ptr;
      uint4 out = make_uint4(0, 0, 0, 0);
      if (r < L) {
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&v);
        __half2 *h = reinterpret_cast<__half2 *>(&out);
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const float2 f = __bfloat1622float2(b[i]);
          h[i] = __floats2half2_rn(f.x, f.y);
        }
      }
      *ptr = out;
    }
  }
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tslot;
  // the first value head of each q/k group publishes the fp16 [K; Q] image for
  // the scan kernel (same layout as its shared-memory operand)
  if (hv % (a.HV / a.H) == 0) {
    constexpr int KQB = kq_image_bytes(DK);
    uint4 *dst = reinterpret_cast<uint4 *>(a.kq_images + ((size_t)slot * a.H + hq) * KQB);
    for (int i = tid; i < KQB / 16; i += kThreads) dst[i] = reinterpret_cast<const uint4 *>(kq)[i];
  }

  // ---- G = [K; Q] K^T ----
  if (tid == 0) {
    const uint32_t sKQ = smem_addr(kq);
    constexpr uint32_t id = idesc_f16(128, C, 0, 0);
#pragma unroll
    for (int k0 = 0; k0 < DK; k0 += 16) {
      const uint64_t d = make_desc(sKQ + (k0 >> 6) * 16384 + (k0 & 63) * 2, 16, 1024);
      mma_f16(tmem, d, d, id, k0 > 0 ? 1u : 0u);  // B = the key rows of the same image
    }
    mma_commit(bar_mma);
  }
  mbar_wait(bar_mma, 0, abort_flag);
  fence_after_sync();

  // ---- A (key lanes) and Aqk (query lanes), decays applied per pair ----
  if (warp * 32 < C) {
    const int r = tid;
    const float br = Gs[r], beta = Bs[r];
#pragma unroll
    for (int s0 = 0; s0 < C; s0 += 16) {
      float g[16];
      tmem_ld16(tmem + lane_base + s0, g);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const int s = s0 + i;
        As[r * LDC + s] = s < r ? beta * g[i] * __expf(br - Gs[s]) : 0.f;
      }
    }
  } else if (warp >= 2 && (warp - 2) * 32 < C) {
    const int r = tid - 64;
    const float br = Gs[r];
    unsigned char *aq = sm + SM::kAqk;
#pragma unroll
    for (int s0 = 0; s0 < C; s0 += 16) {
      float g[16];
      tmem_ld16(tmem + lane_base + s0, g);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 2; h++) {
        uint4 pk;
        __half2 *ph = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const int s = s0 + 8 * h + 2 * i;
          const float v0 = s <= r ? a.scale * g[8 * h + 2 * i] * __expf(br - Gs[s]) : 0.f;
          const float v1 = s + 1 <= r ? a.scale * g[8 * h + 2 * i + 1] * __expf(br - Gs[s + 1]) : 0.f;
          ph[i] = __floats2half2_rn(v0, v1);
        }
        *reinterpret_cast<uint4 *>(aq + kmajor_off(r, s0 + 8 * h, 64)) = pk;
      }
    }
  }
  fence_before_sync();
  __syncthreads();

  // ---- T = (I + A)^-1, in place ----
  constexpr int NB = C / 16;
  {
    float x[16];
    const int I = tid / 16, j = tid % 16, o = 16 * I;
    if (tid < NB * 16) {
#pragma unroll
      for (int r = 0; r < 16; r++) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
      for (int s = 0; s < 16; s++) {
        const float xs = x[s];
#pragma unroll
        for (int r = s + 1; r < 16; r++) x[r] -= As[(o + r) * LDC + o + s] * xs;
      }
    }
    __syncthreads();
    if (tid < NB * 16) {
#pragma unroll
      for (int r = 0; r < 16; r++) As[(o + r) * LDC + o + j] = x[r];
    }
    __syncthreads();
  }
  // block row I: R_J = sum_{K=J}^{I-1} A_IK T_KJ, then T_IJ = -T_II R_J, for
  // J < I; warp J owns column block J (split-bf16 tensor-core products)
  for (int I = 1; I < NB; I++) {
    const int w = 16 * I, J = warp;
    if (J < I) {
      float acc[2][4] = {};
      warp_mma_rt<2, false, false>(
          acc, w - 16 * J, [&](int m, int k) { return As[(w + m) * LDC + 16 * J + k]; },
          [&](int k, int n) { return As[(16 * J + k) * LDC + 16 * J + n]; });
#pragma unroll
      for (int nt = 0; nt < 2; nt++)
#pragma unroll
        for (int e = 0; e < 4; e++) Rs[acc_row(e) * LDC + 16 * J + acc_col(nt, e)] = acc[nt][e];
    }
    __syncthreads();
    if (J < I) {
      float acc[2][4] = {};
      warp_mma<16, 2, false, false>(
          acc, [&](int m, int k) { return As[(w + m) * LDC + w + k]; },
          [&](int k, int n) { return Rs[k * LDC + 16 * J + n]; });
#pragma unroll
      for (int nt = 0; nt < 2; nt++)
#pragma unroll
        for (int e = 0; e < 4; e++) As[(w + acc_row(e)) * LDC + 16 * J + acc_col(nt, e)] = -acc[nt][e];
    }
    __syncthreads();
  }

  // ---- fp16 images of T and D T (MN-major: K-row s holds T[s][0..C)) ----
  if (tid < C) {
    const int s = tid;
    const float d = Ds[s];
#pragma unroll
    for (int ch = 0; ch < C / 8; ch++) {
      uint4 pt, pd;
      __half2 *ht = reinterpret_cast<__half2 *>(&pt);
      __half2 *hd = reinterpret_cast<__half2 *>(&pd);
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float v0 = As[s * LDC + ch * 8 + 2 * i], v1 = As[s * LDC + ch * 8 + 2 * i + 1];
        ht[i] = __floats2half2_rn(v0, v1);
        hd[i] = __floats2half2_rn(d * v0, d * v1);
      }
      *reinterpret_cast<uint4 *>(sm + SM::kTi + mnmajor_chunk_off(s, ch, 64)) = pt;
      *reinterpret_cast<uint4 *>(sm + SM::kDTi + mnmajor_chunk_off(s, ch, 64)) = pd;
    }
  }
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  // ---- P1 = K^T (D T) -> columns [0, C);  AqkT = Aqk T -> columns [64, 64 + C) ----
  if (tid == 0) {
    const uint32_t sKQ = smem_addr(kq), sAqk = smem_addr(sm + SM::kAqk);
    const uint32_t sT = smem_addr(sm + SM::kTi), sDT = smem_addr(sm + SM::kDTi);
    constexpr uint32_t idP = idesc_f16(128, C, 1, 1);   // A MN-major (keys read as K^T)
    constexpr uint32_t idQ = idesc_f16(128, C, 0, 1);
#pragma unroll
    for (int k0 = 0; k0 < C; k0 += 16) {
      const uint64_t ad = make_desc(sKQ + k0 * 128, 16384, 1024);
      const uint64_t bd = make_desc(sDT + (k0 >> 4) * 2048, 8192, 1024);
      mma_f16(tmem, ad, bd, idP, k0 > 0 ? 1u : 0u);
    }
#pragma unroll
    for (int k0 = 0; k0 < C; k0 += 16) {
      const uint64_t ad = make_desc(sAqk + k0 * 2, 16, 1024);
      const uint64_t bd = make_desc(sT + (k0 >> 4) * 2048, 8192, 1024);
      mma_f16(tmem + 64, ad, bd, idQ, k0 > 0 ? 1u : 0u);
    }
    mma_commit(bar_mma);
  }
  mbar_wait(bar_mma, 1, abort_flag);
  fence_after_sync();

  // ---- the image (over the [K; Q] region): row t <- P1 row t, row 128 + t <- AqkT row t ----
  unsigned char *img = kq;
  {
    const int t = tid;
    float v[64];
#pragma unroll
    for (int i = 0; i < 64; i++) v[i] = 0.f;
    if (t < DK) {
#pragma unroll
      for (int s0 = 0; s0 < C; s0 += 16) {
        float g[16];
        tmem_ld16(tmem + lane_base + s0, g);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; i++) v[s0 + i] = g[i];
      }
    }
    // every MMA that read the [K; Q] region is complete; overwrite it
#pragma unroll
    for (int ch = 0; ch < 8; ch++) {
      uint4 pk;
      __half2 *h = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
      for (int i = 0; i < 4; i++) h[i] = __floats2half2_rn(v[ch * 8 + 2 * i], v[ch * 8 + 2 * i + 1]);
      *reinterpret_cast<uint4 *>(img + kmajor_off(t, ch * 8, kPrepImageRows)) = pk;
    }
    if (t < 64) {
#pragma unroll
      for (int i = 0; i < 64; i++) v[i] = 0.f;
      if (warp * 32 < C) {
#pragma unroll
        for (int s0 = 0; s0 < C; s0 += 16) {
          float g[16];
          tmem_ld16(tmem + 64 + lane_base + s0, g);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; i++) v[s0 + i] = g[i];
        }
      }
#pragma unroll
      for (int ch = 0; ch < 8; ch++) {
        uint4 pk;
        __half2 *h = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
        for (int i = 0; i < 4; i++) h[i] = __floats2half2_rn(v[ch * 8 + 2 * i], v[ch * 8 + 2 * i + 1]);
        *reinterpret_cast<uint4 *>(img + kmajor_off(128 + t, ch * 8, kPrepImageRows)) = pk;
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 128);
  uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(a.tiles) +
                                         ((size_t)slot * a.HV + hv) * kPrepImageBytes);
  for (int i = tid; i < kPrepImageBytes / 16; i += kThreads)
    dst[i] = reinterpret_cast<const uint4 *>(img)[i];
  if (*abort_flag && tid == 0) atomicOr(a.flags, kFlagTimeout);
}

template <int C, int DK>
cudaError_t launch_one(const PrepArgs &a, const ScanMaps &maps, cudaStream_t stream) {
  using SM = PrepTmemSmem<C, DK>;
  auto kern = gdn_prep_tmem_kernel<C, DK>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (err != cudaSuccess) return err;
  kern<<<dim3(a.n_slots, a.HV), kThreads, SM::kBytes, stream>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_tmem(const PrepArgs &a, const ScanMaps &maps, int chunk, int dk,
                             cudaStream_t stream) {
  if (chunk == 64 && dk == 128) return launch_one<64, 128>(a, maps, stream);
  if (chunk == 64 && dk == 64) return launch_one<64, 64>(a, maps, stream);
  if (chunk == 32 && dk == 128) return launch_one<32, 128>(a, maps, stream);
  if (chunk == 32 && dk == 64) return launch_one<32, 64>(a, maps, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
