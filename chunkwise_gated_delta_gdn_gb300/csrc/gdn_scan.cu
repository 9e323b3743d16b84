// gdn_scan.cu -- the serial-across-chunks scan kernel of the fp32 path.
//
// One CTA per (sequence, value head, 32-column slice of dv); the slice split
// manufactures parallelism that a (sequence, head) grid lacks (ROCm/rocm-
// libraries PR #11223, "Notes for reviewers": a BH-only scan grid is starved
// below the SM count).  The state slice S (dk x 32, fp32) stays in registers
// as tensor-core accumulators for the whole sequence (the state is
// register-resident in stratat pull #1296, "What this is").  Per chunk, with
// T and Aqk from the prep kernel and S the state at the chunk start:
//
//   gated keys / queries   Kg_r = k_r exp(b_r),  Qg_r = scale q_r exp(b_r)
//   Y      = diag(beta) (V - Kg S)
//   Vn     = T Y                      (= U - W S with U = T diag(beta) V,
//                                       W = T diag(beta) Kg)
//   O      = Qg S + Aqk Vn            -> o (rounded once to the output dtype)
//   S     <- diag(exp(b_last)) S + Kt^T Vn,   Kt_s = k_s exp(b_last - b_s)
//
// (b_last: cumulative gate at the chunk's last row; scalar per row for GDN,
// per key channel for KDA.)  Every product runs on the tensor cores in split
// bf16 (16-bit mantissa operands, fp32 accumulation).  The kernel is written
// for either input type (raw bf16 q/k would be exact operands and skip their
// low halves), but only its fp32 form is compiled.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kScanThreads = 128;
constexpr int NS = kScanSlice;

template <int C, int DK, int GATE>
struct ScanSmem {
  static constexpr int LDK = DK + 4;
  static constexpr int LDC = C + 4;
  static constexpr int LDS = NS + 4;
  static constexpr int kK = 0;                       // keys (gated for KDA)
  static constexpr int kQ = kK + C * LDK;            // queries (gated for KDA)
  static constexpr int kG = kQ + C * LDK;            // KDA: gates -> b -> Kt
  static constexpr int kGsz = GATE == 0 ? 0 : C * LDK;
  static constexpr int kB = kG + kGsz;               // GDN: b, gam, dl (3C)
  static constexpr int kBsz = GATE == 0 ? 3 * C : DK;  // KDA: decay of the chunk
  static constexpr int kBeta = kB + kBsz;
  static constexpr int kV = kBeta + C;
  static constexpr int kT = kV + C * LDS;
  static constexpr int kAqk = kT + C * LDC;
  static constexpr int kS = kAqk + C * LDC;
  static constexpr int kY = kS + DK * LDS;
  static constexpr int kD = kY + C * LDS;            // Vn
  static constexpr int kDD = kD + C * LDS;           // decay-weighted Vn (GDN)
  static constexpr int kO = kDD + C * LDS;           // Qg S partial output
  static constexpr int kFloats = kO + C * LDS;
  static constexpr size_t kBytes = sizeof(float) * kFloats;
  static_assert(C == 32 || C == 64, "the chunk length C is 32 or 64");
  static_assert(DK == 64 || DK == 128, "the key width dk is 64 or 128");
  static_assert(GATE == 0 || GATE == 1, "scalar (GDN) or per-key (KDA) gate");
  static_assert(kBytes <= 227 * 1024, "one CTA's shared memory fits an SM");
};

template <int C, int DK, bool BF16, int GATE>
__global__ void __launch_bounds__(kScanThreads)
gdn_scan_kernel(const ScanArgs a) {
  using SM = ScanSmem<C, DK, GATE>;
  using E = Elem<BF16>;
  extern __shared__ __align__(16) float smem[];
  float *Ks = smem + SM::kK;
  float *Qs = smem + SM::kQ;
  float *Gs = smem + SM::kG;     // KDA only
  float *Bsm = smem + SM::kB;
  float *betas = smem + SM::kBeta;
  float *Vs = smem + SM::kV;
  float *Ts = smem + SM::kT;
  float *Aqks = smem + SM::kAqk;
  float *Ss = smem + SM::kS;
  float *Ys = smem + SM::kY;
  float *Ds = smem + SM::kD;
  float *DDs = smem + SM::kDD;
  float *Os = smem + SM::kO;

  // longest packed sequences first (scan_sequence)
  __shared__ int lpt_pick;
  const int n_slices = a.dv / NS;
  const int hv = (blockIdx.x / n_slices) % a.HV, col0 = (blockIdx.x % n_slices) * NS;
  const int n = scan_sequence(a.seq, blockIdx.x / (a.HV * n_slices), &lpt_pick);
  const int hq = hv / (a.HV / a.H);
  const int tid = threadIdx.x, warp = tid >> 5;

  int start, end;
  bool ok = seq_ok(a.seq, n, start, end);
  if (a.seq.cu) ok = ok && __ldg(a.seq.cu) == 0 && __ldg(a.seq.cu + a.seq.n_seqs) == a.seq.Ttot;
  if (!ok) {
    if (tid == 0) atomicOr(a.flags, kFlagBadSeqlens);
    return;
  }

  // state rows owned by this warp: [r0, r0 + DK/4), MT m-tiles of 16
  constexpr int RW = DK / 4, MT = RW / 16, NT = NS / 8;
  const int r0 = warp * RW;
  float sacc[MT][NT][4];
  const size_t hoff = ((size_t)n * a.HV + hv) * (size_t)DK * a.dv;
#pragma unroll
  for (int mt = 0; mt < MT; mt++)
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int row = r0 + mt * 16 + acc_row(e), col = col0 + acc_col(nt, e);
        sacc[mt][nt][e] = a.h0 ? __ldg(a.h0 + hoff + (size_t)row * a.dv + col) : 0.f;
      }

  const int nchunks = (end - start + C - 1) / C;
  const int base = slot_base<C>(a.seq, n);
  bool nonfinite = false;

  for (int c = 0; c < nchunks; c++) {
    const int t0 = start + c * C;
    const int L = min(C, end - t0);
    const float *tileT = a.tiles + ((size_t)(base + c) * a.HV + hv) * (size_t)(2 * C * C);
    const float *tileAqk = tileT + C * C;
    __syncthreads();  // the previous chunk is done with shared memory

    // ---- loads ----
    load_rows_f32<BF16>(Ks, SM::LDK, static_cast<const typename E::T *>(a.k) +
                            ((long)t0 * a.H + hq) * DK, (long)a.H * DK, C, DK, L);
    load_rows_f32<BF16>(Qs, SM::LDK, static_cast<const typename E::T *>(a.q) +
                            ((long)t0 * a.H + hq) * DK, (long)a.H * DK, C, DK, L);
    load_rows_f32<BF16>(Vs, SM::LDS, static_cast<const typename E::T *>(a.v) +
                            ((long)t0 * a.HV + hv) * a.dv + col0, (long)a.HV * a.dv, C, NS, L);
    for (int idx = tid; idx < C * C / 4; idx += blockDim.x) {
      const int r = idx / (C / 4), c4 = (idx % (C / 4)) * 4;
      *reinterpret_cast<float4 *>(Ts + r * SM::LDC + c4) =
          __ldg(reinterpret_cast<const float4 *>(tileT + r * C + c4));
      *reinterpret_cast<float4 *>(Aqks + r * SM::LDC + c4) =
          __ldg(reinterpret_cast<const float4 *>(tileAqk + r * C + c4));
    }
    for (int r = tid; r < C; r += blockDim.x)
      betas[r] = r < L ? __ldg(a.beta + (long)(t0 + r) * a.HV + hv) : 0.f;
    if constexpr (GATE == 0) {
      for (int r = tid; r < C; r += blockDim.x)
        Bsm[r] = r < L ? __ldg(a.g + (long)(t0 + r) * a.HV + hv) : 0.f;
    } else {
      for (int idx = tid; idx < C * DK / 4; idx += blockDim.x) {
        const int r = idx / (DK / 4), c4 = (idx % (DK / 4)) * 4;
        float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < L) gv = __ldg(reinterpret_cast<const float4 *>(a.g + ((long)(t0 + r) * a.HV + hv) * DK + c4));
        *reinterpret_cast<float4 *>(Gs + r * SM::LDK + c4) = gv;
      }
    }
    // state slice -> shared memory (B operand of the products with S)
#pragma unroll
    for (int mt = 0; mt < MT; mt++)
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int e = 0; e < 4; e++)
          Ss[(r0 + mt * 16 + acc_row(e)) * SM::LDS + acc_col(nt, e)] = sacc[mt][nt][e];
    __syncthreads();

    // ---- gate coefficients ----
    if constexpr (GATE == 0) {
      float *b = Bsm, *gam = Bsm + C, *dl = Bsm + 2 * C;
      if (warp == 0) {
        const int lane = tid & 31;
        float x0 = lane < C ? b[lane] : 0.f;
        float x1 = lane + 32 < C ? b[lane + 32] : 0.f;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const float y0 = __shfl_up_sync(0xffffffffu, x0, d);
          const float y1 = __shfl_up_sync(0xffffffffu, x1, d);
          if (lane >= d) { x0 += y0; x1 += y1; }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        const float blast = __shfl_sync(0xffffffffu, C > 32 ? x1 : x0, (C - 1) & 31);
        if (lane < C) { b[lane] = x0; gam[lane] = __expf(x0); dl[lane] = __expf(blast - x0); }
        if (lane + 32 < C) { b[lane + 32] = x1; gam[lane + 32] = __expf(x1); dl[lane + 32] = __expf(blast - x1); }
      }
    } else {
      // per channel: cumulative gate, then Kt (in place of the gates), and
      // the gated keys / queries in place
      for (int ch = tid; ch < DK; ch += blockDim.x) {
        float run = 0.f;
        for (int r = 0; r < C; r++) {
          run += Gs[r * SM::LDK + ch];
          Gs[r * SM::LDK + ch] = run;
        }
        const float blast = run;
        Bsm[ch] = __expf(blast);
        for (int r = 0; r < C; r++) {
          const float br = Gs[r * SM::LDK + ch];
          const float kv = Ks[r * SM::LDK + ch];
          Gs[r * SM::LDK + ch] = kv * __expf(blast - br);
          const float gr = __expf(br);
          Ks[r * SM::LDK + ch] = kv * gr;
          Qs[r * SM::LDK + ch] = a.scale * Qs[r * SM::LDK + ch] * gr;
        }
      }
    }
    __syncthreads();

    // ---- Kg S -> Y, and Qg S -> partial output ----
    constexpr bool KX = BF16 && GATE == 0;  // raw bf16 keys/queries are exact
    {
      constexpr int NMT = C / 16;
      for (int task = warp; task < 2 * NMT; task += kScanThreads / 32) {
        const int which = task / NMT, m0 = (task % NMT) * 16;
        const float *Am = which == 0 ? Ks : Qs;
        float acc[NT][4] = {};
        warp_mma<DK, NT, KX, false>(
            acc, [&](int m, int k) { return Am[(m0 + m) * SM::LDK + k]; },
            [&](int k, int j) { return Ss[k * SM::LDS + j]; });
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const int r = m0 + acc_row(e), j = acc_col(nt, e);
            if (which == 0) {
              const float x = GATE == 0 ? acc[nt][e] * Bsm[C + r] : acc[nt][e];
              Ys[r * SM::LDS + j] = betas[r] * (Vs[r * SM::LDS + j] - x);
            } else {
              Os[r * SM::LDS + j] = GATE == 0 ? a.scale * Bsm[C + r] * acc[nt][e] : acc[nt][e];
            }
          }
      }
    }
    __syncthreads();

    // ---- Vn = T Y ----
    for (int task = warp; task < C / 16; task += kScanThreads / 32) {
      const int m0 = task * 16;
      float acc[NT][4] = {};
      warp_mma<C, NT, false, false>(
          acc, [&](int m, int k) { return Ts[(m0 + m) * SM::LDC + k]; },
          [&](int k, int j) { return Ys[k * SM::LDS + j]; });
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int r = m0 + acc_row(e), j = acc_col(nt, e);
          Ds[r * SM::LDS + j] = acc[nt][e];
          DDs[r * SM::LDS + j] = GATE == 0 ? acc[nt][e] * Bsm[2 * C + r] : acc[nt][e];
        }
    }
    __syncthreads();

    // ---- O = Qg S + Aqk Vn -> o ----
    for (int task = warp; task < C / 16; task += kScanThreads / 32) {
      const int m0 = task * 16;
      float acc[NT][4] = {};
      warp_mma<C, NT, false, false>(
          acc, [&](int m, int k) { return Aqks[(m0 + m) * SM::LDC + k]; },
          [&](int k, int j) { return Ds[k * SM::LDS + j]; });
      typename E::T *orow = static_cast<typename E::T *>(a.o);
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int r = m0 + acc_row(e), j = acc_col(nt, e);
          if (r < L) {
            const float v0 = Os[r * SM::LDS + j] + acc[nt][e];
            const float v1 = Os[r * SM::LDS + j + 1] + acc[nt][e + 1];
            nonfinite |= !(isfinite(v0) && isfinite(v1));
            typename E::T *dst = orow + ((long)(t0 + r) * a.HV + hv) * a.dv + col0 + j;
            dst[0] = E::from_f(v0);
            dst[1] = E::from_f(v1);
          }
        }
    }

    // ---- S <- diag(decay) S + Kt^T Vn ----
    {
      const float *Kt = GATE == 0 ? Ks : Gs;
#pragma unroll
      for (int mt = 0; mt < MT; mt++) {
        const int m0 = r0 + mt * 16;
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const float dec = GATE == 0 ? Bsm[C + C - 1] : Bsm[m0 + acc_row(e)];
            sacc[mt][nt][e] *= dec;
          }
        warp_mma<C, NT, KX, false>(
            sacc[mt], [&](int m, int k) { return Kt[k * SM::LDK + m0 + m]; },
            [&](int k, int j) { return DDs[k * SM::LDS + j]; });
      }
    }
  }

  // ---- final state ----
  if (a.hT) {
#pragma unroll
    for (int mt = 0; mt < MT; mt++)
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int row = r0 + mt * 16 + acc_row(e), col = col0 + acc_col(nt, e);
          const float v = sacc[mt][nt][e];
          nonfinite |= !isfinite(v);
          a.hT[hoff + (size_t)row * a.dv + col] = v;
        }
  }
  if (__syncthreads_or(nonfinite) && tid == 0) atomicOr(a.flags, kFlagNonfinite);
}

template <int C, int DK, bool BF16, int GATE>
cudaError_t launch_one(const ScanArgs &a, cudaStream_t stream) {
  using SM = ScanSmem<C, DK, GATE>;
  auto kern = gdn_scan_kernel<C, DK, BF16, GATE>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SM::kBytes);
  if (err != cudaSuccess) return err;
  const long blocks = (long)a.seq.n_seqs * a.HV * (a.dv / NS);
  if (blocks > 0x7fffffffL) return cudaErrorInvalidValue;
  kern<<<(unsigned)blocks, kScanThreads, SM::kBytes, stream>>>(a);
  return cudaGetLastError();
}

// Instantiated for fp32 inputs only: bf16 inputs run the tensor-memory
// kernels, so the bf16 form of this kernel is not compiled.
template <int C, int DK>
cudaError_t dispatch_dt_gate(const ScanArgs &a, int dtype, int gate, cudaStream_t s) {
  if (dtype == 0 && gate == 0) return launch_one<C, DK, false, 0>(a, s);
  if (dtype == 0 && gate == 1) return launch_one<C, DK, false, 1>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_scan(const ScanArgs &a, int chunk, int dk, int dtype, int gate,
                        cudaStream_t stream) {
  if (chunk == 64 && dk == 128) return dispatch_dt_gate<64, 128>(a, dtype, gate, stream);
  if (chunk == 64 && dk == 64) return dispatch_dt_gate<64, 64>(a, dtype, gate, stream);
  if (chunk == 32 && dk == 128) return dispatch_dt_gate<32, 128>(a, dtype, gate, stream);
  if (chunk == 32 && dk == 64) return dispatch_dt_gate<32, 64>(a, dtype, gate, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
