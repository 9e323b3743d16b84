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
// Convolution layout: one thread owns 4 adjacent channels (one 8-byte bf16
// load per token) and walks 128 consecutive tokens, keeping the last W - 1
// inputs in registers; a warp covers 128 channels of a token with coalesced
// 256-byte accesses, and loads eight tokens ahead of use.  Four channels keep
// the thread under 80 registers, so that enough warps share an SM to cover
// the memory latency.  A tile re-reads only its W - 1 tokens of halo.  The
// norms give each row 32 (L2) or 16 (gated RMS) lanes, each lane a contiguous
// piece of it, and load all of a warp's rows before the first is reduced.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;
constexpr int kConvVec = 4;      // channels per thread
constexpr int kConvTokens = 128;  // tokens per thread (halo re-read: W - 1 of them)
constexpr int kConvAhead = 8;    // tokens loaded ahead of use

// 4 consecutive elements, raw: one 8-byte load for bf16, one 16-byte for fp32
template <bool BF16>
struct Raw4;
template <>
struct Raw4<true> {
  uint2 u;
};
template <>
struct Raw4<false> {
  uint4 u;
};
template <bool BF16>
__device__ __forceinline__ Raw4<BF16> load_raw4(const void *base, size_t elem) {
  Raw4<BF16> r;
  if constexpr (BF16)
    r.u = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(base) + elem));
  else
    r.u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const float *>(base) + elem));
  return r;
}
template <bool BF16>
__device__ __forceinline__ void unpack4(const Raw4<BF16> &r, float (&v)[4]) {
  if constexpr (BF16) {
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.u.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.u.y));
    v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
  } else {
    v[0] = __uint_as_float(r.u.x); v[1] = __uint_as_float(r.u.y);
    v[2] = __uint_as_float(r.u.z); v[3] = __uint_as_float(r.u.w);
  }
}
template <bool BF16>
__device__ __forceinline__ void load4(const void *base, size_t elem, float (&v)[4]) {
  unpack4<BF16>(load_raw4<BF16>(base, elem), v);
}
template <bool BF16>
__device__ __forceinline__ void store4(void *base, size_t elem, const float (&v)[4]) {
  if constexpr (BF16) {
    const __nv_bfloat162 b0 = __floats2bfloat162_rn(v[0], v[1]);
    const __nv_bfloat162 b1 = __floats2bfloat162_rn(v[2], v[3]);
    *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(base) + elem) =
        make_uint2(*reinterpret_cast<const uint32_t *>(&b0), *reinterpret_cast<const uint32_t *>(&b1));
  } else {
    *reinterpret_cast<float4 *>(static_cast<float *>(base) + elem) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// SiLU with the fast exponential and division intrinsics: relative error a few
// units of 2^-22 for |x| < 10, far inside one rounding to bf16 (2^-9)
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }

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

// SPLIT: the launch covers the token tiles from a.tile0 on (inputs of more
// than 65535 tiles, the grid's y extent, take several launches); the common
// form keeps the tile index a pure function of blockIdx.y, which compiles
// to faster code
template <int W, bool BF16, bool SILU, bool SPLIT>
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
  const int tt0 = SPLIT ? (a.tile0 + (int)blockIdx.y) * kConvTokens : (int)blockIdx.y * kConvTokens;
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
      load4<BF16>(a.x, (size_t)tau * a.D + c0, xv);
#pragma unroll
      for (int v = 0; v < kConvVec; v++) win[i][v] = xv[v];
    } else {
#pragma unroll
      for (int v = 0; v < kConvVec; v++) win[i][v] = hist(n, tt0 - start + i, v);
    }
  }
#pragma unroll 1
  for (int tb = tt0; tb < tt1; tb += kConvAhead) {
    // the next kConvAhead tokens' inputs in flight together
    Raw4<BF16> raw[kConvAhead];
#pragma unroll
    for (int u = 0; u < kConvAhead; u++)
      if (tb + u < tt1) raw[u] = load_raw4<BF16>(a.x, (size_t)(tb + u) * a.D + c0);
#pragma unroll
    for (int u = 0; u < kConvAhead; u++) {
      const int t = tb + u;
      if (t >= tt1) break;
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
      unpack4<BF16>(raw[u], xv);
#pragma unroll
      for (int v = 0; v < kConvVec; v++) {
        float acc = bs[v];
#pragma unroll
        for (int i = 0; i < H; i++) acc = fmaf(wt[i][v], win[i][v], acc);
        acc = fmaf(wt[W - 1][v], xv[v], acc);
        out[v] = SILU ? silu(acc) : acc;
      }
      store4<BF16>(a.y, (size_t)t * a.D + c0, out);
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
// row norms: LPR lanes per row (32 or 16), lane l of a row owns elements
// [l E, l E + E), E = DIM / LPR
// ---------------------------------------------------------------------------
// a lane's E contiguous elements as 32-bit words, in the widest aligned
// vector loads (E 16-bit or 32-bit elements = E/2 or E words)
template <int NW>
__device__ __forceinline__ void ld_words(const uint32_t *p, uint32_t (&w)[NW]) {
  if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 4) {
      const uint4 u = *reinterpret_cast<const uint4 *>(p + i);
      w[i] = u.x; w[i + 1] = u.y; w[i + 2] = u.z; w[i + 3] = u.w;
    }
  } else if constexpr (NW % 2 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 2) {
      const uint2 u = *reinterpret_cast<const uint2 *>(p + i);
      w[i] = u.x; w[i + 1] = u.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < NW; i++) w[i] = p[i];
  }
}
template <int NW>
__device__ __forceinline__ void st_words(uint32_t *p, const uint32_t (&w)[NW]) {
  if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 4)
      *reinterpret_cast<uint4 *>(p + i) = make_uint4(w[i], w[i + 1], w[i + 2], w[i + 3]);
  } else if constexpr (NW % 2 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 2) *reinterpret_cast<uint2 *>(p + i) = make_uint2(w[i], w[i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < NW; i++) p[i] = w[i];
  }
}

template <int E, bool BF16>
__device__ __forceinline__ void load_row(const void *base, size_t off, float (&v)[E]) {
  if constexpr (BF16) {
    uint32_t w[E / 2];
    ld_words<E / 2>(reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(base) + off), w);
#pragma unroll
    for (int i = 0; i < E / 2; i++) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  } else {
    uint32_t w[E];
    ld_words<E>(reinterpret_cast<const uint32_t *>(static_cast<const float *>(base) + off), w);
#pragma unroll
    for (int i = 0; i < E; i++) v[i] = __uint_as_float(w[i]);
  }
}

template <int E, bool BF16>
__device__ __forceinline__ void store_row(void *base, size_t off, const float (&v)[E]) {
  if constexpr (BF16) {
    uint32_t w[E / 2];
#pragma unroll
    for (int i = 0; i < E / 2; i++) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
    st_words<E / 2>(reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(base) + off), w);
  } else {
    uint32_t w[E];
#pragma unroll
    for (int i = 0; i < E; i++) w[i] = __float_as_uint(v[i]);
    st_words<E>(reinterpret_cast<uint32_t *>(static_cast<float *>(base) + off), w);
  }
}

// LPR lanes per row, so 32 / LPR rows side by side in a warp, and RPW such
// row groups per warp, all loaded before the first is reduced, so that each
// lane keeps several loads in flight.  Rows past the end load zeros and are
// not stored; every lane takes the same path (the row sums are warp
// shuffles).  KIND 0: L2 norm; 1: gated RMS norm.
template <int DIM, bool BF16, int KIND, int RPW, int LPR>
__global__ void __launch_bounds__(256) gdn_rownorm_kernel(RowNormArgs a) {
  constexpr int E = DIM / LPR, RG = 32 / LPR;
  const int lane = threadIdx.x & 31, l = lane % LPR;
  const long row0 = (blockIdx.x * 8L + (threadIdx.x >> 5)) * (RPW * RG) + lane / LPR;
  float v[RPW][E], z[RPW][E];
#pragma unroll
  for (int q = 0; q < RPW; q++) {
    const long row = row0 + q * RG;
    if (row < a.rows) {
      const size_t off = (size_t)row * DIM + l * E;
      load_row<E, BF16>(a.x, off, v[q]);
      if (KIND == 1 && a.z) load_row<E, BF16>(a.z, off, z[q]);
    } else {
#pragma unroll
      for (int i = 0; i < E; i++) v[q][i] = z[q][i] = 0.f;
    }
  }
#pragma unroll
  for (int q = 0; q < RPW; q++) {
    const long row = row0 + q * RG;
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < E; i++) s = fmaf(v[q][i], v[q][i], s);
#pragma unroll
    for (int d = LPR / 2; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
    if constexpr (KIND == 0) {
      const float r = rsqrtf(s + a.eps);
#pragma unroll
      for (int i = 0; i < E; i++) v[q][i] *= r;
    } else {
      const float r = rsqrtf(s * (1.f / DIM) + a.eps);
#pragma unroll
      for (int i = 0; i < E; i++) {
        v[q][i] = v[q][i] * r * __ldg(a.weight + l * E + i);
        if (a.z) v[q][i] *= silu(z[q][i]);
      }
    }
    if (row < a.rows) store_row<E, BF16>(a.y, (size_t)row * DIM + l * E, v[q]);
  }
}

template <int W, bool BF16>
cudaError_t conv_w(const ConvArgs &a, int act, cudaStream_t s) {
  // token tiles on the grid's y axis, at most 65535 per launch (one launch
  // below 8.4 M tokens)
  const long tiles = ((long)a.seq.Ttot + kConvTokens - 1) / kConvTokens;
  const bool split = tiles > 65535;
  for (long t0 = 0; t0 < tiles; t0 += 65535) {
    ConvArgs b = a;
    b.tile0 = (int)t0;
    const dim3 grid((a.D / kConvVec + kConvThreads - 1) / kConvThreads,
                    (unsigned)(tiles - t0 < 65535 ? tiles - t0 : 65535));
    if (split)
      (act ? gdn_conv1d_kernel<W, BF16, true, true> : gdn_conv1d_kernel<W, BF16, false, true>)
          <<<grid, kConvThreads, 0, s>>>(b);
    else
      (act ? gdn_conv1d_kernel<W, BF16, true, false> : gdn_conv1d_kernel<W, BF16, false, false>)
          <<<grid, kConvThreads, 0, s>>>(b);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.hT && W > 1) {
    const long n = (long)a.seq.n_seqs * a.D;
    gdn_conv1d_state_kernel<W, BF16><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

template <int DIM, bool BF16, int KIND, int RPW, int LPR>
void rows_launch(const RowNormArgs &a, cudaStream_t s) {
  constexpr long per = 8L * RPW * (32 / LPR);  // rows per CTA of 8 warps
  gdn_rownorm_kernel<DIM, BF16, KIND, RPW, LPR><<<(unsigned)((a.rows + per - 1) / per), 256, 0, s>>>(a);
}

template <int DIM, bool BF16>
cudaError_t rows_dim(const RowNormArgs &a, int kind, cudaStream_t s) {
  // L2: a warp per row, four rows per warp in turn.  Gated RMS (two input
  // streams and a SiLU per element): 16 lanes per row with the widest loads,
  // two rows side by side, one pair per warp (at 32k tokens x 48 heads: 195
  // against 222 us with a warp per row and two rows in turn; two or four
  // pairs per warp, or 8 lanes per row, were slower)
  if (kind == 0)
    rows_launch<DIM, BF16, 0, 4, 32>(a, s);
  else
    rows_launch<DIM, BF16, 1, 1, 16>(a, s);
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
  if (a.rows > 16L * 0x7fffffffL) return cudaErrorInvalidValue;  // grid.x extent
  return dtype == 1 ? rows_dt<true>(a, dim, kind, stream) : rows_dt<false>(a, dim, kind, stream);
}

}  // namespace gdn
