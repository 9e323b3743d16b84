// gdn_prep.cu -- the state-independent chunk-prep kernel of the fp32 path.
//
// One CTA per (chunk slot, value head).  For the C-row chunk it forms
//   b      cumulative natural-log gates (per key channel for KDA)
//   A      = strict-lower(beta_r * sum_c k_rc k_sc exp(b_rc - b_sc))
//   Aqk    = lower-incl-diag(scale * sum_c q_rc k_sc exp(b_rc - b_sc))
//   T      = (I + A)^-1, unit lower triangular, by a blocked solve
// and writes T and Aqk (fp32, C x C each) to the workspace tile of the slot.
// These are the state-independent tiles of ROCm/rocm-libraries PR #11223
// ("Summary": A and Aqk; "Levers" 3: blocked triangular solve with scalar
// forward substitution inside each diagonal block and rank updates against the
// solved blocks).  The gated-key and gated-query tiles (GK, GQ, Kt, dec) are
// cheap elementwise products and are formed by the scan kernel when it needs
// them, so they never cross HBM.
//
// GDN: the Gram K K^T and Q K^T run on the tensor cores (split-bf16 operands,
// fp32 accumulation); the scalar pairwise decay exp(b_r - b_s) is applied per
// element afterwards, never factored, and only for s <= r, so no exponent is
// positive.  KDA: the per-channel decay sits inside the contraction; each
// pair (r, s <= r) is summed by one warp over the channels with the exponent
// difference formed directly (no midpoint factoring), which is exact in range
// for any gate <= 0.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kPrepThreads = 256;

template <int C, int DK, int GATE>
struct PrepSmem {
  static constexpr int LDK = DK + 4;  // fp32 row stride of the K / Q tiles
  static constexpr int LDC = C + 4;   // fp32 row stride of the C x C tiles
  static constexpr int LDG = GATE == 0 ? 1 : LDK;
  static constexpr int kK = 0;
  static constexpr int kQ = kK + C * LDK;
  static constexpr int kG = kQ + C * LDK;          // gates, then cumulative gates
  static constexpr int kBeta = kG + C * LDG;
  static constexpr int kA = kBeta + C;
  static constexpr int kT = kA + C * LDC;
  static constexpr int kR = kT + C * LDC;          // 16 x 17 scratch of the solve
  static constexpr int kMeta = kR + 16 * 17;       // t0, L, valid
  static constexpr int kFloats = kMeta + 4;
  static constexpr size_t kBytes = sizeof(float) * kFloats;
  static_assert(C == 32 || C == 64, "the chunk length C is 32 or 64");
  static_assert(DK == 64 || DK == 128, "the key width dk is 64 or 128");
  static_assert(GATE == 0 || GATE == 1, "scalar (GDN) or per-key (KDA) gate");
  static_assert(kBytes <= 227 * 1024, "one CTA's shared memory fits an SM");
};

template <int C, int DK, bool BF16, int GATE>
__global__ void __launch_bounds__(kPrepThreads)
gdn_prep_kernel(const PrepArgs a) {
  using SM = PrepSmem<C, DK, GATE>;
  extern __shared__ __align__(16) float smem[];
  float *Ks = smem + SM::kK;
  float *Qs = smem + SM::kQ;
  float *Gs = smem + SM::kG;
  float *Bs = smem + SM::kBeta;
  float *As = smem + SM::kA;
  float *Ts = smem + SM::kT;
  float *Rs = smem + SM::kR;
  int *meta = reinterpret_cast<int *>(smem + SM::kMeta);

  const int slot = blockIdx.x;
  const int hv = blockIdx.y;
  const int hq = hv / (a.HV / a.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- which sequence and chunk this slot belongs to (binary search) ----
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

  // ---- loads: K, Q (fp32 copies), gates, beta ----
  load_rows_f32<BF16>(Ks, SM::LDK, static_cast<const typename Elem<BF16>::T *>(a.k) +
                          ((long)t0 * a.H + hq) * DK, (long)a.H * DK, C, DK, L);
  load_rows_f32<BF16>(Qs, SM::LDK, static_cast<const typename Elem<BF16>::T *>(a.q) +
                          ((long)t0 * a.H + hq) * DK, (long)a.H * DK, C, DK, L);
  bool positive = false;
  if constexpr (GATE == 0) {
    for (int r = tid; r < C; r += blockDim.x) {
      const float gv = r < L ? __ldg(a.g + (long)(t0 + r) * a.HV + hv) : 0.f;
      positive |= gv > 0.f;
      Gs[r] = gv;
    }
  } else {
    for (int idx = tid; idx < C * DK / 4; idx += blockDim.x) {
      const int r = idx / (DK / 4), c4 = (idx % (DK / 4)) * 4;
      float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < L) gv = __ldg(reinterpret_cast<const float4 *>(a.g + ((long)(t0 + r) * a.HV + hv) * DK + c4));
      positive |= (gv.x > 0.f) | (gv.y > 0.f) | (gv.z > 0.f) | (gv.w > 0.f);
      *reinterpret_cast<float4 *>(Gs + r * SM::LDG + c4) = gv;
    }
  }
  for (int r = tid; r < C; r += blockDim.x)
    Bs[r] = r < L ? __ldg(a.beta + (long)(t0 + r) * a.HV + hv) : 0.f;
  if (__syncthreads_or(positive) && tid == 0) atomicOr(a.flags, kFlagPositiveGate);

  // ---- cumulative log-gates (in place) ----
  if constexpr (GATE == 0) {
    if (warp == 0) {
      // inclusive scan of C <= 64 values: two per lane
      float x0 = lane < C ? Gs[lane] : 0.f;
      float x1 = lane + 32 < C ? Gs[lane + 32] : 0.f;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, x0, d);
        const float y1 = __shfl_up_sync(0xffffffffu, x1, d);
        if (lane >= d) { x0 += y0; x1 += y1; }
      }
      x1 += __shfl_sync(0xffffffffu, x0, 31);
      if (lane < C) Gs[lane] = x0;
      if (lane + 32 < C) Gs[lane + 32] = x1;
    }
  } else {
    for (int c = tid; c < DK; c += blockDim.x) {
      float run = 0.f;
      for (int r = 0; r < C; r++) {
        run += Gs[r * SM::LDG + c];
        Gs[r * SM::LDG + c] = run;
      }
    }
  }
  // T starts as zero (its strictly upper blocks stay zero)
  for (int idx = tid; idx < C * SM::LDC; idx += blockDim.x) Ts[idx] = 0.f;
  __syncthreads();

  float *tileT = a.tiles + ((size_t)slot * a.HV + hv) * (size_t)(2 * C * C);
  float *tileAqk = tileT + C * C;

  // ---- A and Aqk ----
  if constexpr (GATE == 0) {
    // tasks: {K K^T, Q K^T} x (C/16 row tiles) x (C/32 column groups of 32)
    constexpr int NMT = C / 16, NNG = C / 32, NTASK = 2 * NMT * NNG;
    for (int task = warp; task < NTASK; task += kPrepThreads / 32) {
      const int which = task / (NMT * NNG);
      const int mt = (task / NNG) % NMT, ng = task % NNG;
      const int m0 = mt * 16, n0 = ng * 32;
      float acc[4][4] = {};
      if (n0 <= m0 + 15) {  // tiles fully above the diagonal are zero
        const float *Am = which == 0 ? Ks : Qs;
        warp_mma<DK, 4, BF16, BF16>(
            acc, [&](int m, int k) { return Am[(m0 + m) * SM::LDK + k]; },
            [&](int k, int n) { return Ks[(n0 + n) * SM::LDK + k]; });
      }
#pragma unroll
      for (int nt = 0; nt < 4; nt++) {
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int r = m0 + acc_row(e);
          const int s = n0 + acc_col(nt, e);
          float v0 = 0.f, v1 = 0.f;
          if (which == 0) {
            if (s < r) v0 = Bs[r] * acc[nt][e] * __expf(Gs[r] - Gs[s]);
            if (s + 1 < r) v1 = Bs[r] * acc[nt][e + 1] * __expf(Gs[r] - Gs[s + 1]);
            As[r * SM::LDC + s] = v0;
            As[r * SM::LDC + s + 1] = v1;
          } else {
            if (s <= r) v0 = a.scale * acc[nt][e] * __expf(Gs[r] - Gs[s]);
            if (s + 1 <= r) v1 = a.scale * acc[nt][e + 1] * __expf(Gs[r] - Gs[s + 1]);
            *reinterpret_cast<float2 *>(tileAqk + r * C + s) = make_float2(v0, v1);
          }
        }
      }
    }
  } else {
    // one warp per pair (r, s <= r); lanes stride over the key channels
    constexpr int NPAIR = C * (C + 1) / 2;
    for (int p = warp; p < NPAIR; p += kPrepThreads / 32) {
      int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
      while ((r + 1) * (r + 2) / 2 <= p) r++;
      while (r * (r + 1) / 2 > p) r--;
      const int s = p - r * (r + 1) / 2;
      float kk = 0.f, qk = 0.f;
      for (int c = lane; c < DK; c += 32) {
        const float d = __expf(Gs[r * SM::LDG + c] - Gs[s * SM::LDG + c]);
        const float ks = Ks[s * SM::LDK + c] * d;
        kk += Ks[r * SM::LDK + c] * ks;
        qk += Qs[r * SM::LDK + c] * ks;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        kk += __shfl_xor_sync(0xffffffffu, kk, off);
        qk += __shfl_xor_sync(0xffffffffu, qk, off);
      }
      if (lane == 0) {
        As[r * SM::LDC + s] = s < r ? Bs[r] * kk : 0.f;
        tileAqk[r * C + s] = a.scale * qk;
      }
    }
    // upper triangles: A and Aqk are zero there
    for (int idx = tid; idx < C * C; idx += blockDim.x) {
      const int r = idx / C, s = idx % C;
      if (s > r) {
        As[r * SM::LDC + s] = 0.f;
        tileAqk[idx] = 0.f;
      }
    }
  }
  __syncthreads();

  // ---- blocked solve T = (I + A)^-1 ----
  constexpr int NB = C / 16;
  // diagonal blocks: forward substitution, one thread per (block, column)
  if (tid < NB * 16) {
    const int I = tid / 16, j = tid % 16, o = 16 * I;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; r++) {
      float v = (r == j) ? 1.f : 0.f;
#pragma unroll
      for (int s = 0; s < r; s++) v -= As[(o + r) * SM::LDC + o + s] * x[s];
      x[r] = v;
    }
#pragma unroll
    for (int r = 0; r < 16; r++) Ts[(o + r) * SM::LDC + o + j] = x[r];
  }
  __syncthreads();
  // off-diagonal blocks by distance d = I - J:
  //   R = sum_{K=J}^{I-1} A_IK T_KJ,   T_IJ = -T_II R
  for (int d = 1; d < NB; d++) {
    for (int I = d; I < NB; I++) {
      const int J = I - d;
      {
        const int m = tid >> 4, j = tid & 15;
        float acc = 0.f;
        for (int s = 16 * J; s < 16 * I; s++)
          acc += As[(16 * I + m) * SM::LDC + s] * Ts[s * SM::LDC + 16 * J + j];
        Rs[m * 17 + j] = acc;
      }
      __syncthreads();
      {
        const int m = tid >> 4, j = tid & 15;
        float acc = 0.f;
        for (int p = 0; p <= m; p++)
          acc += Ts[(16 * I + m) * SM::LDC + 16 * I + p] * Rs[p * 17 + j];
        Ts[(16 * I + m) * SM::LDC + 16 * J + j] = -acc;
      }
      __syncthreads();
    }
  }

  // ---- write T ----
  for (int idx = tid; idx < C * C / 4; idx += blockDim.x) {
    const int r = idx / (C / 4), c4 = (idx % (C / 4)) * 4;
    *reinterpret_cast<float4 *>(tileT + r * C + c4) =
        *reinterpret_cast<const float4 *>(Ts + r * SM::LDC + c4);
  }
}

template <int C, int DK, bool BF16, int GATE>
cudaError_t launch_one(const PrepArgs &a, cudaStream_t stream) {
  using SM = PrepSmem<C, DK, GATE>;
  auto kern = gdn_prep_kernel<C, DK, BF16, GATE>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SM::kBytes);
  if (err != cudaSuccess) return err;
  dim3 grid(a.n_slots, a.HV);
  kern<<<grid, kPrepThreads, SM::kBytes, stream>>>(a);
  return cudaGetLastError();
}

// Instantiated for fp32 inputs only: bf16 inputs run the tensor-memory
// kernels, so the bf16 form of this kernel is not compiled.
template <int C, int DK>
cudaError_t dispatch_dt_gate(const PrepArgs &a, int dtype, int gate, cudaStream_t s) {
  if (dtype == 0 && gate == 0) return launch_one<C, DK, false, 0>(a, s);
  if (dtype == 0 && gate == 1) return launch_one<C, DK, false, 1>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prep(const PrepArgs &a, int chunk, int dk, int dtype, int gate,
                        cudaStream_t stream) {
  if (chunk == 64 && dk == 128) return dispatch_dt_gate<64, 128>(a, dtype, gate, stream);
  if (chunk == 64 && dk == 64) return dispatch_dt_gate<64, 64>(a, dtype, gate, stream);
  if (chunk == 32 && dk == 128) return dispatch_dt_gate<32, 128>(a, dtype, gate, stream);
  if (chunk == 32 && dk == 64) return dispatch_dt_gate<32, 64>(a, dtype, gate, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
