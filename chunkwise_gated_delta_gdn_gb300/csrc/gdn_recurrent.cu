// gdn_recurrent.cu -- the token-serial (recurrent) form of the gated delta
// rule: one token at a time with the state held in registers.  With T == 1 it
// is the decode step (logismos issue #46, "Verified implementation boundary":
// a one-token grouped step with K-first input state and separate output and
// next-state buffers); with T > 1 it walks the tokens of each sequence in
// order, which is the plain definition the chunked kernels reproduce.
//
// Per token t, value head hv, q/k head hq = hv / (HV / H), state S (dk x dv,
// fp32, K-first):
//     S   <- diag(a) S                 a = exp(g_t): one scalar (GDN) or one
//                                      value per key channel (KDA)
//     u   =  beta_t (v_t - S^T k_t)    (dv)
//     o_t =  scale (S^T q_t + (k_t . q_t) u)   = scale (S + k_t u^T)^T q_t
//     S   <- S + k_t u^T
// The read uses the updated state without forming it first: S^T q and S^T k
// come out of one pass over the decayed state, and k.q closes the rank-1 term.
//
// The work is bound by the state's HBM traffic (read dk x dv fp32 once, write
// it once per call); everything else is a few hundred bytes per (token, head).
// One CTA of 128 threads owns a (sequence, value head, 32-column slice): lane
// (w, l) holds the dk/16 consecutive rows from dk/16 (4 w + l/8) on, columns
// 4 (l % 8) .. +3.  Every 8 lanes read one 128-byte row segment (coalesced
// float4 loads and stores of the state), a thread's pieces of k, q and the
// per-key gates are contiguous (16-byte loads), and the column sums over rows
// reduce by two shuffles and one pass over shared memory.  A thread holds 128
// bytes of state at dk = 128, and seven (per-key gate, 72 registers) or eight
// (scalar gate, 64) CTAs fit on an SM: 112-128 KB of loads in flight per SM,
// enough to keep HBM busy through each CTA's load -> reduce -> store
// sequence.  Measured on one decode step of 256 sequences (dk = dv = 128):
// with 256 threads of 4 rows each (five CTAs per SM, 80 KB) the scalar-gate
// step ran at 86% of the copy bandwidth; with 8 rows per thread 16 rows apart
// (scalar loads of k, q and the gates) at 96% (scalar gate) and 80% (per-key
// gate); with the rows contiguous at 98% and 95%.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kRecThreads = 128;
constexpr int kRecSlice = 32;  // dv columns per CTA

// N consecutive elements (bf16 or fp32) as floats, in 16-byte loads (one
// 8-byte load for 4 bf16 elements); the address aligned to the load's size
template <int N, bool BF16>
__device__ __forceinline__ void load_vec(const void *p, float (&v)[N]) {
  if constexpr (BF16) {
    static_assert(N % 8 == 0 || N == 4, "whole 16- or 8-byte pieces");
    if constexpr (N % 8 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 8) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p) + i));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[j]));
          v[i + 2 * j] = f.x; v[i + 2 * j + 1] = f.y;
        }
      }
    } else {
      const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
      const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
      const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
      v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
    }
  } else {
    static_assert(N % 4 == 0, "whole 16-byte pieces");
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const float4 f = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i));
      v[i] = f.x; v[i + 1] = f.y; v[i + 2] = f.z; v[i + 3] = f.w;
    }
  }
}

template <int DK, bool BF16, int GATE>
__global__ void __launch_bounds__(kRecThreads) gdn_recurrent_kernel(RecurrentArgs a) {
  using E = Elem<BF16>;
  using T = typename E::T;
  constexpr int NW = kRecThreads / 32;
  constexpr int RPT = DK / (4 * NW);  // rows per thread
  const int n = blockIdx.x, hv = blockIdx.y, j0 = blockIdx.z * kRecSlice;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, cg = lane & 7;
  const int r0 = (w * 4 + (lane >> 3)) * RPT;  // this thread's rows: r0 .. r0 + RPT - 1
  const int hq = hv / (a.HV / a.H);

  __shared__ float red[NW][8][9];  // [warp][column group][4 x S^T k, 4 x S^T q, k.q]
  __shared__ __align__(16) float ub[kRecSlice];

  int start, end;
  bool ok = seq_ok(a.seq, n, start, end);
  if (a.seq.cu) ok = ok && __ldg(a.seq.cu) == 0 && __ldg(a.seq.cu + a.seq.n_seqs) == a.seq.Ttot;
  if (!ok) {  // uniform across the block
    if (tid == 0 && a.flags) atomicOr(a.flags, kFlagBadSeqlens);
    return;
  }

  // the state slice; plain loads (hT may be h0: this block writes back exactly
  // the elements it read, and no other block touches them)
  const size_t sbase = ((size_t)n * a.HV + hv) * DK * (size_t)a.dv + j0 + 4 * cg;
  float4 S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; i++) {
    if (a.h0)
      S[i] = *reinterpret_cast<const float4 *>(a.h0 + sbase + (size_t)(r0 + i) * a.dv);
    else
      S[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  const T *qp = static_cast<const T *>(a.q);
  const T *kp = static_cast<const T *>(a.k);
  const T *vp = static_cast<const T *>(a.v);
  T *op = static_cast<T *>(a.o);
  bool positive = false, nonfinite = false;

  for (int t = start; t < end; t++) {
    const size_t qk = ((size_t)t * a.H + hq) * DK + r0;
    const size_t th = (size_t)t * a.HV + hv;
    float kk[RPT], qq[RPT], dec[RPT];
    load_vec<RPT, BF16>(kp + qk, kk);
    load_vec<RPT, BF16>(qp + qk, qq);
    if constexpr (GATE == 0) {
      const float gt = __ldg(a.g + th);
      positive |= gt > 0.f;
      const float d = expf(gt);
#pragma unroll
      for (int i = 0; i < RPT; i++) dec[i] = d;
    } else {
      float gt[RPT];
      load_vec<RPT, false>(a.g + th * DK + r0, gt);
#pragma unroll
      for (int i = 0; i < RPT; i++) {
        positive |= gt[i] > 0.f;
        dec[i] = expf(gt[i]);
      }
    }
    const float bt = __ldg(a.beta + th);

    // decay, then this thread's share of S^T k, S^T q and k.q
    float p[9];
#pragma unroll
    for (int e = 0; e < 9; e++) p[e] = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; i++) {
      S[i].x *= dec[i]; S[i].y *= dec[i]; S[i].z *= dec[i]; S[i].w *= dec[i];
      p[0] = fmaf(S[i].x, kk[i], p[0]);
      p[1] = fmaf(S[i].y, kk[i], p[1]);
      p[2] = fmaf(S[i].z, kk[i], p[2]);
      p[3] = fmaf(S[i].w, kk[i], p[3]);
      p[4] = fmaf(S[i].x, qq[i], p[4]);
      p[5] = fmaf(S[i].y, qq[i], p[5]);
      p[6] = fmaf(S[i].z, qq[i], p[6]);
      p[7] = fmaf(S[i].w, qq[i], p[7]);
      p[8] = fmaf(kk[i], qq[i], p[8]);
    }
    // sum over the 4 row groups of the warp (lanes 8 and 16 apart)
#pragma unroll
    for (int e = 0; e < 9; e++) {
      p[e] += __shfl_xor_sync(0xffffffffu, p[e], 8);
      p[e] += __shfl_xor_sync(0xffffffffu, p[e], 16);
    }
    if (lane < 8) {
#pragma unroll
      for (int e = 0; e < 9; e++) red[w][cg][e] = p[e];
    }
    __syncthreads();
    if (tid < kRecSlice) {  // one thread per column of the slice
      const int c = tid >> 2, e = tid & 3;
      float sk = 0.f, sq = 0.f, kq = 0.f;
#pragma unroll
      for (int ww = 0; ww < NW; ww++) {
        sk += red[ww][c][e];
        sq += red[ww][c][4 + e];
        kq += red[ww][0][8];
      }
      const size_t vo = th * (size_t)a.dv + j0 + tid;
      const float u = bt * (E::to_f(vp[vo]) - sk);
      const float ot = a.scale * fmaf(kq, u, sq);
      ub[tid] = u;
      const T ob = E::from_f(ot);
      nonfinite |= !isfinite(E::to_f(ob));
      op[vo] = ob;
    }
    __syncthreads();
    const float4 u4 = reinterpret_cast<const float4 *>(ub)[cg];
#pragma unroll
    for (int i = 0; i < RPT; i++) {
      S[i].x = fmaf(kk[i], u4.x, S[i].x);
      S[i].y = fmaf(kk[i], u4.y, S[i].y);
      S[i].z = fmaf(kk[i], u4.z, S[i].z);
      S[i].w = fmaf(kk[i], u4.w, S[i].w);
    }
  }

  if (a.hT) {
#pragma unroll
    for (int i = 0; i < RPT; i++) {
      nonfinite |= !(isfinite(S[i].x) && isfinite(S[i].y) && isfinite(S[i].z) &&
                     isfinite(S[i].w));
      *reinterpret_cast<float4 *>(a.hT + sbase + (size_t)(r0 + i) * a.dv) = S[i];
    }
  }
  if (a.flags) {
    const uint32_t bits = (positive ? kFlagPositiveGate : 0u) | (nonfinite ? kFlagNonfinite : 0u);
    if (bits) atomicOr(a.flags, bits);
  }
}

template <int DK, bool BF16, int GATE>
cudaError_t launch_one(const RecurrentArgs &a, cudaStream_t stream) {
  const dim3 grid(a.seq.n_seqs, a.HV, a.dv / kRecSlice);
  gdn_recurrent_kernel<DK, BF16, GATE><<<grid, kRecThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const RecurrentArgs &a, int dtype, int gate, cudaStream_t stream) {
  if (dtype == 1)
    return gate == 0 ? launch_one<DK, true, 0>(a, stream) : launch_one<DK, true, 1>(a, stream);
  return gate == 0 ? launch_one<DK, false, 0>(a, stream) : launch_one<DK, false, 1>(a, stream);
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentArgs &a, int dk, int dtype, int gate,
                             cudaStream_t stream) {
  if (a.seq.n_seqs <= 0 || a.dv % kRecSlice != 0) return cudaErrorInvalidValue;
  if (dk == 64) return launch_dk<64>(a, dtype, gate, stream);
  if (dk == 128) return launch_dk<128>(a, dtype, gate, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
