// gdn_device.cuh -- device helpers shared by the prep and scan kernels:
// sequence/slot mapping, tile loads, and a warp-level split-bf16 tensor-core
// product that keeps fp32-class precision.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_internal.h"

namespace gdn {

// ---------------------------------------------------------------------------
// sequences and chunk slots
// ---------------------------------------------------------------------------
__device__ __forceinline__ int seq_start(const SeqInfo &s, int n) {
  return s.cu ? __ldg(s.cu + n) : n * s.T;
}

template <int C>
__device__ __forceinline__ int slot_base(const SeqInfo &s, int n) {
  return seq_start(s, n) / C + n;
}

// Validity of packed sequence n: 0 <= start <= end <= Ttot.
__device__ __forceinline__ bool seq_ok(const SeqInfo &s, int n, int &start,
                                       int &end) {
  start = seq_start(s, n);
  end = seq_start(s, n + 1);
  return start >= 0 && start <= end && end <= s.Ttot;
}

// Block order of the serial scans.  Blocks are launched in index order, and a
// block runs one (sequence, value head, dv slice) chain from start to end, so
// block b = rank * HV * slices + head * slices + slice, where for packed input
// of up to kLptSeqs sequences the rank counts sequences by decreasing length
// (ties by index): the longest chains start first and the short ones fill in
// behind them (greedy longest-first list scheduling).  Otherwise rank =
// sequence.  Every thread of the block calls this (it synchronises the
// block); `pick` is one int of shared memory.
constexpr int kLptSeqs = 64;
__device__ __forceinline__ int scan_sequence(const SeqInfo &s, int rank, int *pick) {
  if (!s.cu || s.n_seqs > kLptSeqs) return rank;
  for (int i = threadIdx.x; i < s.n_seqs; i += blockDim.x) {
    const int li = __ldg(s.cu + i + 1) - __ldg(s.cu + i);
    int longer = 0;
    for (int j = 0; j < s.n_seqs; j++) {
      const int lj = __ldg(s.cu + j + 1) - __ldg(s.cu + j);
      longer += (lj > li || (lj == li && j < i)) ? 1 : 0;
    }
    if (longer == rank) *pick = i;  // exactly one i: the order is strict
  }
  __syncthreads();
  return *pick;
}

// ---------------------------------------------------------------------------
// element conversion
// ---------------------------------------------------------------------------
template <bool BF16>
struct Elem;
template <>
struct Elem<true> {
  using T = __nv_bfloat16;
  static __device__ __forceinline__ float to_f(T x) { return __bfloat162float(x); }
  static __device__ __forceinline__ T from_f(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Elem<false> {
  using T = float;
  static __device__ __forceinline__ float to_f(T x) { return x; }
  static __device__ __forceinline__ T from_f(float x) { return x; }
};

// Load `rows` x `cols` of a row-major global matrix (row stride `gstride`
// elements) into fp32 shared memory (row stride `sstride` floats); rows at or
// beyond `valid` are zero.  cols must be a multiple of 8.
template <bool BF16>
__device__ __forceinline__ void load_rows_f32(float *dst, int sstride,
                                              const void *src, long gstride,
                                              int rows, int cols, int valid) {
  using E = Elem<BF16>;
  const typename E::T *s = reinterpret_cast<const typename E::T *>(src);
  const int per_row = cols / 8;
  for (int idx = threadIdx.x; idx < rows * per_row; idx += blockDim.x) {
    const int r = idx / per_row, c8 = (idx % per_row) * 8;
    float vals[8];
    if (r < valid) {
      if constexpr (BF16) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(s + r * gstride + c8));
        const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
        for (int e = 0; e < 8; e++) vals[e] = __bfloat162float(b[e]);
      } else {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(s + r * gstride + c8));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(s + r * gstride + c8 + 4));
        vals[0] = a.x; vals[1] = a.y; vals[2] = a.z; vals[3] = a.w;
        vals[4] = b.x; vals[5] = b.y; vals[6] = b.z; vals[7] = b.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; e++) vals[e] = 0.f;
    }
    float *d = dst + r * sstride + c8;
    *reinterpret_cast<float4 *>(d) = make_float4(vals[0], vals[1], vals[2], vals[3]);
    *reinterpret_cast<float4 *>(d + 4) = make_float4(vals[4], vals[5], vals[6], vals[7]);
  }
}

// ---------------------------------------------------------------------------
// split-bf16 warp MMA
//
// An fp32 operand x is carried as hi = bf16(x), lo = bf16(x - hi): 16
// mantissa bits.  A product of two fp32 operands is hi*hi + hi*lo + lo*hi
// (lo*lo, below 2^-32 relative, is dropped); an operand known to be exactly
// bf16 (an unmodified bf16 input) has lo = 0 and skips its terms.  All
// accumulation is fp32 on the tensor cores (mma.sync m16n8k16).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 lo_idx, __nv_bfloat16 hi_idx) {
  return (static_cast<uint32_t>(__bfloat16_as_ushort(hi_idx)) << 16) |
         static_cast<uint32_t>(__bfloat16_as_ushort(lo_idx));
}

__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  const __nv_bfloat16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
  const __nv_bfloat16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
  hi = pack_bf16(h0, h1);
  lo = pack_bf16(l0, l1);
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc[nt] (a 16 x 8*NT fp32 tile, mma accumulator layout) += A * B with
// A: 16 x KDIM, B: KDIM x 8*NT.  a_at(m, k) and b_at(k, n) return fp32
// elements relative to the tile origin.  AX / BX: operand exactly bf16.
template <int KDIM, int NT, bool AX, bool BX, typename FA, typename FB>
__device__ __forceinline__ void warp_mma(float (&acc)[NT][4], FA a_at, FB b_at) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
#pragma unroll 1
  for (int k0 = 0; k0 < KDIM; k0 += 16) {
    uint32_t ahi[4], alo[4];
    split2(a_at(gq, k0 + 2 * tq), a_at(gq, k0 + 2 * tq + 1), ahi[0], alo[0]);
    split2(a_at(gq + 8, k0 + 2 * tq), a_at(gq + 8, k0 + 2 * tq + 1), ahi[1], alo[1]);
    split2(a_at(gq, k0 + 2 * tq + 8), a_at(gq, k0 + 2 * tq + 9), ahi[2], alo[2]);
    split2(a_at(gq + 8, k0 + 2 * tq + 8), a_at(gq + 8, k0 + 2 * tq + 9), ahi[3], alo[3]);
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      const int n = nt * 8 + gq;
      uint32_t bhi0, blo0, bhi1, blo1;
      split2(b_at(k0 + 2 * tq, n), b_at(k0 + 2 * tq + 1, n), bhi0, blo0);
      split2(b_at(k0 + 2 * tq + 8, n), b_at(k0 + 2 * tq + 9, n), bhi1, blo1);
      if constexpr (!AX) mma16816(acc[nt], alo, bhi0, bhi1);
      if constexpr (!BX) mma16816(acc[nt], ahi, blo0, blo1);
      mma16816(acc[nt], ahi, bhi0, bhi1);
    }
  }
}

// As warp_mma, with the contraction length `kdim` (a multiple of 16) known
// only at run time.
template <int NT, bool AX, bool BX, typename FA, typename FB>
__device__ __forceinline__ void warp_mma_rt(float (&acc)[NT][4], int kdim, FA a_at, FB b_at) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
#pragma unroll 1
  for (int k0 = 0; k0 < kdim; k0 += 16) {
    uint32_t ahi[4], alo[4];
    split2(a_at(gq, k0 + 2 * tq), a_at(gq, k0 + 2 * tq + 1), ahi[0], alo[0]);
    split2(a_at(gq + 8, k0 + 2 * tq), a_at(gq + 8, k0 + 2 * tq + 1), ahi[1], alo[1]);
    split2(a_at(gq, k0 + 2 * tq + 8), a_at(gq, k0 + 2 * tq + 9), ahi[2], alo[2]);
    split2(a_at(gq + 8, k0 + 2 * tq + 8), a_at(gq + 8, k0 + 2 * tq + 9), ahi[3], alo[3]);
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      const int n = nt * 8 + gq;
      uint32_t bhi0, blo0, bhi1, blo1;
      split2(b_at(k0 + 2 * tq, n), b_at(k0 + 2 * tq + 1, n), bhi0, blo0);
      split2(b_at(k0 + 2 * tq + 8, n), b_at(k0 + 2 * tq + 9, n), bhi1, blo1);
      if constexpr (!AX) mma16816(acc[nt], alo, bhi0, bhi1);
      if constexpr (!BX) mma16816(acc[nt], ahi, blo0, blo1);
      mma16816(acc[nt], ahi, bhi0, bhi1);
    }
  }
}

// ---------------------------------------------------------------------------
// split-tf32 warp MMA (m16n8k8): x = hi + lo with hi = tf32(x), lo = tf32(x - hi)
// (about 21 mantissa bits); a product is lo*hi + hi*lo + hi*hi, accumulated in
// fp32 on the tensor cores.  Operands come straight from registers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
  uint32_t h, l;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(x));
  const float r = x - __uint_as_float(h);
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(l) : "f"(r));
  hi = h;
  lo = l;
}

__device__ __forceinline__ void mma1688_tf32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc (a 16 x 8 fp32 tile, accumulator layout) += A B over k = k0 .. k0 + 7,
// a_at(m, k) and b_at(k, n) giving fp32 elements relative to the tile origin.
// The hi*hi terms go to `acc`, the two correction terms to `corr` (added to
// acc by the caller at the end), so the three products of a step do not wait
// on one another.
template <typename FA, typename FB>
__device__ __forceinline__ void warp_mma_tf32x3(float (&acc)[4], float (&corr)[4], int k0,
                                                FA a_at, FB b_at) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  uint32_t ah[4], al[4], bh0, bl0, bh1, bl1;
  split_tf32(a_at(gq, k0 + tq), ah[0], al[0]);
  split_tf32(a_at(gq + 8, k0 + tq), ah[1], al[1]);
  split_tf32(a_at(gq, k0 + tq + 4), ah[2], al[2]);
  split_tf32(a_at(gq + 8, k0 + tq + 4), ah[3], al[3]);
  split_tf32(b_at(k0 + tq, gq), bh0, bl0);
  split_tf32(b_at(k0 + tq + 4, gq), bh1, bl1);
  mma1688_tf32(acc, ah, bh0, bh1);
  mma1688_tf32(corr, al, bh0, bh1);
  mma1688_tf32(corr, ah, bl0, bl1);
}

// ---------------------------------------------------------------------------
// one-pass fp16 warp MMA (m16n8k16): operands rounded once to fp16 (11
// significand bits), products accumulated in fp32 on the tensor cores.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_f16(float lo_elem, float hi_elem) {
  const __half2 h = __floats2half2_rn(lo_elem, hi_elem);
  return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void mma16816_f16(float (&c)[4], const uint32_t (&a)[4],
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc (a 16 x 8 fp32 tile, accumulator layout) += A B over k = k0 .. k0 + 15;
// a_at(m, k) and b_at(k, n) give fp32 elements relative to the tile origin.
template <typename FA, typename FB>
__device__ __forceinline__ void warp_mma_f16(float (&acc)[4], int k0, FA a_at, FB b_at) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  const int k = k0 + 2 * tq;
  uint32_t a[4];
  a[0] = pack_f16(a_at(gq, k), a_at(gq, k + 1));
  a[1] = pack_f16(a_at(gq + 8, k), a_at(gq + 8, k + 1));
  a[2] = pack_f16(a_at(gq, k + 8), a_at(gq, k + 9));
  a[3] = pack_f16(a_at(gq + 8, k + 8), a_at(gq + 8, k + 9));
  const uint32_t b0 = pack_f16(b_at(k, gq), b_at(k + 1, gq));
  const uint32_t b1 = pack_f16(b_at(k + 8, gq), b_at(k + 9, gq));
  mma16816_f16(acc, a, b0, b1);
}

// Row / column of accumulator element e of n-tile nt for this lane.
__device__ __forceinline__ int acc_row(int e) { return ((threadIdx.x & 31) >> 2) + ((e & 2) ? 8 : 0); }
__device__ __forceinline__ int acc_col(int nt, int e) { return nt * 8 + 2 * (threadIdx.x & 3) + (e & 1); }

}  // namespace gdn
