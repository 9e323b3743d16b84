// gdn_prepost.cu -- the operations either side of the gated delta rule, each
// a memory-bound CUDA kernel:
//
//  * causal depthwise convolution over time with a raw-input history (the
//    staged causal convolution of logismos issue #46, "Verified
//    implementation boundary": channel-major oldest-to-newest history,
//    separate next-history and output, no history for width 1).  For channel
//    c, width W and ext = [history; x] of one sequence,
//        y[t, c] = act(bias[c] + sum_j w[c, j] ext[t + j]),   act = id or SiLU,
//    and the next history is the last W - 1 entries of ext;
//  * L2 normalisation of rows (the unit-norm q and k the recurrence expects):
//        y = x / sqrt(sum(x^2) + eps);
//  * gated RMS normalisation of output rows (the output norm that follows the
//    recurrence, stratat pull #1296, re-base notes):
//        y = x / sqrt(mean(x^2) + eps) * weight [* silu(z)].
//
// Convolution layout: one thread owns 8 adjacent channels (one 16-byte bf16
// load per token) and walks 32 consecutive tokens, keeping the last W - 1
// inputs in registers; a warp covers 256 channels of a token with coalesced
// 512-byte accesses.  A tile re-reads only its W - 1 tokens of halo.  The
// norms give one warp to a row, each lane a contiguous piece of it.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;
constexpr int kConvVec = 8;      // channels per thread
constexpr int kConvTokens = 32;  // tokens per thread

template <bool BF16>
__device__ __forceinline__ void load8(const void *base, size_t elem, float (&v)[8]) {
  if constexpr (BF16) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
        static_cast<const __nv_bfloat16 *>(base) + elem));
    const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const float2 f = __bfloat1622float2(b[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  } else {
    const float *p = static_cast<const float *>(base) + elem;
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

template <bool BF16>
__device__ __forceinline__ void store8(void *base, size_t elem, const float (&v)[8]) {
  if constexpr (BF16) {
    uint4 raw;
    __nv_bfloat162 *b = reinterpret_cast<__nv_bfloat162 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; i++) b[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(base) + elem) = raw;
  } else {
    float *p = static_cast<float *>(base) + elem;
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
  }
}

__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

// sequence holding token `tok` (largest n with start_n <= tok), or -1
__device__ __forceinline__ int seq_of(const SeqInfo &s, int tok) {
  if (!s.cu) return s.T > 0 ? tok / s.T : -1;
  int lo = 0, hi = s.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(s.cu + mid) <= tok) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// every cu_seqlens entry a block may visit is checked here: 0 = c0 <= c1 <=
// .. <= cN = Ttot
__device__ bool seqlens_ok(const SeqInfo &s) {
  if (!s.cu) return true;
  if (__ldg(s.cu) != 0 || __ldg(s.cu + s.n_seqs) != s.Ttot) return false;
  for (int n = 0; n < s.n_seqs; n++)
    if (__ldg(s.cu + n) > __ldg(s.cu + n + 1)) return false;
  return true;
}

template <int W, bool BF16, bool SILU>
__global__ void __launch_bounds__(kConvThreads) gdn_conv1d_kernel(ConvArgs a) {
  __shared__ int ok_s;
  if (threadIdx.x == 0) ok_s = seqlens_ok(a.seq) ? 1 : 0;
  __syncthreads();
  if (!ok_s) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && a.flags)
      atomicOr(a.flags, kFlagBadSeqlens);
    return;
  }
  const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * kConvVec;
  const int tt0 = blockIdx.y * kConvTokens;
  if (c0 >= a.D || tt0 >= a.seq.Ttot) return;
  const int tt1 = min(tt0 + kConvTokens, a.seq.Ttot);
  constexpr int H = W - 1;  // history length

  float wt[W][kConvVec], bs[kConvVec];
#pragma unroll
  for (int v = 0; v < kConvVec; v++) {
#pragma unroll
    for (int j = 0; j < W; j++) wt[j][v] = __ldg(a.w + (size_t)(c0 + v) * W + j);
    bs[v] = a.bias ? __ldg(a.bias + c0 + v) : 0.f;
  }
  // the window: win[i] = input i + 1 - W tokens before the current one
  float win[H > 0 ? H : 1][kConvVec];
  int n = seq_of(a.seq, tt0);
  int start = seq_start(a.seq, n), end = seq_start(a.seq, n + 1);
  auto hist = [&](int seq, int i, int v) -> float {
    return a.h0 ? __ldg(a.h0 + ((size_t)seq * a.D + c0 + v) * (H > 0 ? H : 1) + i) : 0.f;
  };
  // inputs before the tile's first token: from x inside the sequence, else
  // from the sequence's history
#pragma unroll
  for (int i = 0; i < H; i++) {
    const int tau = tt0 - H + i;
    if (tau >= start) {
      float xv[kConvVec];
      load8<BF16>(a.x, (size_t)tau * a.D + c0, xv);
#pragma unroll
      for (int v = 0; v < kConvVec; v++) win[i][v] = xv[v];
    } else {
#pragma unroll
      for (int v = 0; v < kConvVec; v++) win[i][v] = hist(n, tt0 - start + i, v);
    }
  }
  for (int t = tt0; t < tt1; t++) {
    if (t >= end) {  // the next non-empty sequence starts at t
      while (t >= end && n + 1 < a.seq.n_seqs) {
        n++;
        start = end;
        end = seq_start(a.seq, n + 1);
      }
#pragma unroll
      for (int i = 0; i < H; i++)
#pragma unroll
        for (int v = 0; v < kConvVec; v++) win[i][v] = hist(n, i, v);
    }
    float xv[kConvVec], out[kConvVec];
    load8<BF16>(a.x, (size_t)t * a.D + c0, xv);
#pragma unroll
    for (int v = 0; v < kConvVec; v++) {
      float acc = bs[v];
#pragma unroll
      for (int i = 0; i < H; i++) acc = fmaf(wt[i][v], win[i][v], acc);
      acc = fmaf(wt[W - 1][v], xv[v], acc);
      out[v] = SILU ? silu(acc) : acc;
    }
    store8<BF16>(a.y, (size_t)t * a.D + c0, out);
#pragma unroll
    for (int i = 0; i + 1 < H; i++)
#pragma unroll
      for (int v = 0; v < kConvVec; v++) win[i][v] = win[i + 1][v];
    if constexpr (H > 0) {
#pragma unroll
      for (int v = 0; v < kConvVec; v++) win[H - 1][v] = xv[v];
    }
  }
}

// next history: hT[n, c, i] = ext[L + i] of sequence n (ext = [h0; x]); one
// thread per (sequence, channel).  Runs after the convolution, so hT may be
// h0 itself (each thread reads index i + L >= i before writing index i).
template <int W, bool BF16>
__global__ void __launch_bounds__(256) gdn_conv1d_state_kernel(ConvArgs a) {
  constexpr int H = W - 1;
  const long idx = blockIdx.x * 256L + threadIdx.x;
  if (idx >= (long)a.seq.n_seqs * a.D) return;
  const int n = (int)(idx / a.D), c = (int)(idx % a.D);
  int start, end;
  if (!seq_ok(a.seq, n, start, end)) return;  // flagged by the convolution
  const int L = end - start;
  for (int i = 0; i < H; i++) {
    float val;
    if (i + L < H) {
      val = a.h0 ? a.h0[((size_t)n * a.D + c) * H + i + L] : 0.f;
    } else {
      const size_t e = (size_t)(end - H + i) * a.D + c;
      if constexpr (BF16)
        val = __bfloat162float(static_cast<const __nv_bfloat16 *>(a.x)[e]);
      else
        val = static_cast<const float *>(a.x)[e];
    }
    a.hT[((size_t)n * a.D + c) * H + i] = val;
  }
}

// ---------------------------------------------------------------------------
// row norms: one warp per row, lane l owns elements [l E, l E + E), E = DIM/32
// ---------------------------------------------------------------------------
template <int E, bool BF16>
__device__ __forceinline__ void load_row(const void *base, size_t off, float (&v)[E]) {
  if constexpr (BF16) {
    const __nv_bfloat16 *p = static_cast<const __nv_bfloat16 *>(base) + off;
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p + i));
      v[i] = f.x;
      v[i + 1] = f.y;
    }
  } else {
    const float *p = static_cast<const float *>(base) + off;
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const float2 f = *reinterpret_cast<const float2 *>(p + i);
      v[i] = f.x;
      v[i + 1] = f.y;
    }
  }
}

template <int E, bool BF16>
__device__ __forceinline__ void store_row(void *base, size_t off, const float (&v)[E]) {
  if constexpr (BF16) {
    __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(base) + off;
#pragma unroll
    for (int i = 0; i < E; i += 2)
      *reinterpret_cast<__nv_bfloat162 *>(p + i) = __floats2bfloat162_rn(v[i], v[i + 1]);
  } else {
    float *p = static_cast<float *>(base) + off;
#pragma unroll
    for (int i = 0; i < E; i += 2) *reinterpret_cast<float2 *>(p + i) = make_float2(v[i], v[i + 1]);
  }
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
  return s;
}

template <int DIM, bool BF16>
__global__ void __launch_bounds__(256) gdn_l2norm_kernel(RowNormArgs a) {
  constexpr int E = DIM / 32;
  const long row = blockIdx.x * 8L + (threadIdx.x >> 5);
  if (row >= a.rows) return;
  const int lane = threadIdx.x & 31;
  const size_t off = (size_t)row * DIM + lane * E;
  float v[E];
  load_row<E, BF16>(a.x, off, v);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < E; i++) s = fmaf(v[i], v[i], s);
  const float r = rsqrtf(warp_sum(s) + a.eps);
#pragma unroll
  for (int i = 0; i < E; i++) v[i] *= r;
  store_row<E, BF16>(a.y, off, v);
}

template <int DIM, bool BF16>
__global__ void __launch_bounds__(256) gdn_rmsnorm_gated_kernel(RowNormArgs a) {
  constexpr int E = DIM / 32;
  const long row = blockIdx.x * 8L + (threadIdx.x >> 5);
  if (row >= a.rows) return;
  const int lane = threadIdx.x & 31;
  const size_t off = (size_t)row * DIM + lane * E;
  float v[E];
  load_row<E, BF16>(a.x, off, v);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < E; i++) s = fmaf(v[i], v[i], s);
  const float r = rsqrtf(warp_sum(s) * (1.f / DIM) + a.eps);
  float z[E];
  if (a.z) load_row<E, BF16>(a.z, off, z);
#pragma unroll
  for (int i = 0; i < E; i++) {
    v[i] = v[i] * r * __ldg(a.weight + lane * E + i);
    if (a.z) v[i] *= silu(z[i]);
  }
  store_row<E, BF16>(a.y, off, v);
}

template <int W, bool BF16>
cudaError_t conv_w(const ConvArgs &a, int act, cudaStream_t s) {
  const dim3 grid((a.D / kConvVec + kConvThreads - 1) / kConvThreads,
                  (a.seq.Ttot + kConvTokens - 1) / kConvTokens);
  if (a.seq.Ttot > 0) {
    if (act)
      gdn_conv1d_kernel<W, BF16, true><<<grid, kConvThreads, 0, s>>>(a);
    else
      gdn_conv1d_kernel<W, BF16, false><<<grid, kConvThreads, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.hT && W > 1) {
    const long n = (long)a.seq.n_seqs * a.D;
    gdn_conv1d_state_kernel<W, BF16><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

template <int DIM, bool BF16>
cudaError_t rows_dim(const RowNormArgs &a, int kind, cudaStream_t s) {
  const unsigned grid = (unsigned)((a.rows + 7) / 8);
  if (kind == 0)
    gdn_l2norm_kernel<DIM, BF16><<<grid, 256, 0, s>>>(a);
  else
    gdn_rmsnorm_gated_kernel<DIM, BF16><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <bool BF16>
cudaError_t rows_dt(const RowNormArgs &a, int dim, int kind, cudaStream_t s) {
  switch (dim) {
    case 64: return rows_dim<64, BF16>(a, kind, s);
    case 128: return rows_dim<128, BF16>(a, kind, s);
    case 256: return rows_dim<256, BF16>(a, kind, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_conv1d(const ConvArgs &a, int width, int activation, int dtype,
                          cudaStream_t stream) {
  if (a.D % kConvVec != 0) return cudaErrorInvalidValue;
  const bool bf = dtype == 1;
  switch (width) {
    case 1: return bf ? conv_w<1, true>(a, activation, stream) : conv_w<1, false>(a, activation, stream);
    case 2: return bf ? conv_w<2, true>(a, activation, stream) : conv_w<2, false>(a, activation, stream);
    case 3: return bf ? conv_w<3, true>(a, activation, stream) : conv_w<3, false>(a, activation, stream);
    case 4: return bf ? conv_w<4, true>(a, activation, stream) : conv_w<4, false>(a, activation, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rownorm(const RowNormArgs &a, int dim, int kind, int dtype,
                           cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  return dtype == 1 ? rows_dt<true>(a, dim, kind, stream) : rows_dt<false>(a, dim, kind, stream);
}

}  // namespace gdn
