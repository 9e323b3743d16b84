// gdn_prep_tc.cu -- the state-independent chunk-prep kernel of the bf16
// per-key-gate (KDA) path.  (The scalar gate runs gdn_prep_tmem.cu.)
//
// One CTA (128 threads) per (chunk slot, value head).  From the chunk's keys,
// queries, gates and beta it forms, in fp32:
//   b      cumulative natural-log gates, per key channel
//   A      = strict-lower(beta_r sum_c k_rc k_sc exp(b_rc - b_sc))
//   Aqk    = lower-incl-diag(scale sum_c q_rc k_sc exp(b_rc - b_sc))
//   T      = (I + A)^-1   (blocked: 16 x 16 diagonal blocks by forward
//            substitution, then block rows by products against the solved
//            blocks; ROCm/rocm-libraries PR #11223, "Levers" 3)
//   P1     = Kt^T T       (Kt_s = k_s exp(b_last - b_s); dk x C)
//   AqkT   = Aqk T        (C x C)
// and writes P1 and AqkT (tcgen05 products of fp16 operands, fp32 accumulation
// in tensor memory), rounded once to fp16, as one 24 KB operand image in
// the scan kernel's shared-memory layout (K-major, 128-byte swizzle, 192 rows
// of 64 elements: rows 0..127 = P1 (rows >= dk zero), rows 128..191 = AqkT,
// columns >= C zero).  With Y = diag(beta)(V - Kg S) the scan then needs only
//   S <- diag(exp(b_last)) S + P1 Y     and     O = Qg S + AqkT Y,
// the WY products W = T diag(beta) Kg and U = T diag(beta) V of stratat pull
// #1296 ("What this is") folded into P1 and AqkT so that no dk-wide W ever
// crosses HBM.  It also publishes the scan's gated operand image [Kg; Qg]
// (Kg = k e^b, Qg = scale q e^b, fp16) and the chunk's per-channel decay
// e^{b_last}.  The factored A / Aqk products run on the tensor cores in split
// bf16 (mma.sync, 16 significant bits and the fp32 range their factors need);
// P1 and Aqk T, whose operands stay within fp16, run as tcgen05 products like
// the scalar-gate path's.  The image is stored with one bulk copy.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;

template <int C, int DK>
struct PrepTcSmem {
  static constexpr int LDB = DK + 8;  // bf16 row stride of K / Q
  static constexpr int LDC = C + 4;   // fp32 row stride of C x C tiles
  static constexpr int LDG = DK + 4;
  // byte offsets
  static constexpr int kK = 0;
  static constexpr int kQ = kK + C * LDB * 2;  // Q, then (with A) the image
  static constexpr int QSZ = (C * LDB * 2 + C * LDC * 4 >= kPrepImageBytes)
                                 ? C * LDB * 2
                                 : kPrepImageBytes - C * LDC * 4;
  static constexpr int kA = kQ + QSZ;
  static constexpr int kImgSpan = QSZ + C * LDC * 4;  // Q + A regions
  static constexpr int kAqk = kA + C * LDC * 4;
  static constexpr int kT = kAqk + C * LDC * 4;
  static constexpr int kR = kT + C * LDC * 4;                  // 16 x LDC scratch
  static constexpr int kG = kR + 16 * LDC * 4;                 // gates -> b -> Kt
  static constexpr int kBeta = kG + C * LDG * 4;
  static constexpr int kMeta = kBeta + C * 4;
  // factored operands of one 16-row block, each split into bf16 hi and lo
  // planes (x = hi + lo, 16 significant bits, the fp32 exponent range):
  // K~ hi, K~ lo, Q~ hi, Q~ lo (16 rows each), then K^ hi, K^ lo (C rows
  // each); bf16 row stride LDH (a 16-byte multiple, rows 272 bytes apart so
  // that ldmatrix's eight row reads fall in different banks)
  static constexpr int LDH = DK + 8;
  static constexpr int kBar = (kMeta + 16 + 7) / 8 * 8;      // the products' mbarrier
  static constexpr int kTslot = kBar + 8;                    // tensor-memory address
  static constexpr int kAbort = kTslot + 4;
  static constexpr int kX = (kAbort + 4 + 1023) / 1024 * 1024;
  static constexpr int XBYTES = (4 * 16 + 2 * C) * LDH * 2;
  // Once A and Aqk are formed, the X region holds the fp16 operands of the
  // image products (K-major, 128-byte swizzle): Kt as C token rows x dk in
  // two 64-channel panels (read MN-major: M = dk), T as C rows (row j =
  // column j of T), Aqk as 128 rows (rows >= C not written; their products
  // are not read)
  static constexpr int kOpKt = kX;
  static constexpr int kOpT = kOpKt + 2 * C * 128;
  static constexpr int kOpAqk = kOpT + C * 128;
  static constexpr int kBytes = kX + (XBYTES > 2 * C * 128 + C * 128 + 128 * 128
                                          ? XBYTES : 2 * C * 128 + C * 128 + 128 * 128) + 1024;
  static_assert(kImgSpan >= kPrepImageBytes, "image must fit the Q + A regions");
  static_assert(kX % 1024 == 0 && kOpT % 1024 == 0 && kOpAqk % 1024 == 0, "operand alignment");
};

// four 8 x 8 bf16 matrices (x4) / two (x2) from rows of shared memory: lane l
// gives the address of one row (mma.sync fragment order)
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t &r0, uint32_t &r1, uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(saddr));
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi), four values at a time
__device__ __forceinline__ void split4(float4 x, uint2 &hi, uint2 &lo) {
  split2(x.x, x.y, hi.x, lo.x);
  split2(x.z, x.w, hi.y, lo.y);
}


template <int C, int DK>
__global__ void __launch_bounds__(kThreads)
gdn_prep_tc_kernel(const PrepArgs a) {
  using SM = PrepTcSmem<C, DK>;
  extern __shared__ unsigned char smem_raw[];
  // 1 KB-aligned base (the tensor-core operands use the 128-byte swizzle)
  unsigned char *smem = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
  __nv_bfloat16 *Kb = reinterpret_cast<__nv_bfloat16 *>(smem + SM::kK);
  __nv_bfloat16 *Qb = reinterpret_cast<__nv_bfloat16 *>(smem + SM::kQ);
  float *As = reinterpret_cast<float *>(smem + SM::kA);
  float *Aqks = reinterpret_cast<float *>(smem + SM::kAqk);
  float *Ts = reinterpret_cast<float *>(smem + SM::kT);
  float *Rs = reinterpret_cast<float *>(smem + SM::kR);
  float *Gs = reinterpret_cast<float *>(smem + SM::kG);
  float *Bs = reinterpret_cast<float *>(smem + SM::kBeta);
  int *meta = reinterpret_cast<int *>(smem + SM::kMeta);
  unsigned char *img = smem + SM::kQ;  // valid once Q and A are dead

  const int slot = blockIdx.x, hv = blockIdx.y;
  const int hq = hv / (a.HV / a.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int LDB = SM::LDB, LDC = SM::LDC, LDG = SM::LDG;

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
  if (!meta[2]) return;
  const int t0 = meta[0], L = meta[1];
  // tensor memory for the image products: P1 at column 0, Aqk T at 64
  constexpr uint32_t kTmemCols = 128;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + SM::kTslot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM::kAbort);
  const uint32_t bar_mma = sm100::smem_addr(smem + SM::kBar);
  if (warp == 0) sm100::tmem_alloc(sm100::smem_addr(tslot), kTmemCols);
  if (tid == 0) {
    *abort_flag = 0;
    sm100::mbar_init(bar_mma, 1);
    sm100::mbar_fence_init();
  }

  // ---- loads ----
  {
    const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(a.k) + ((long)t0 * a.H + hq) * DK;
    const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(a.q) + ((long)t0 * a.H + hq) * DK;
    // asynchronous copies, all in flight at once; rows past the chunk's
    // tokens are zero-filled
    constexpr int PER = DK / 8;
    for (int idx = tid; idx < C * PER; idx += kThreads) {
      const int r = idx / PER, c8 = (idx % PER) * 8;
      const bool in = r < L;
      const long off = (in ? (long)r * a.H * DK : 0) + c8;
      sm100::cp_async16(sm100::smem_addr(Kb + r * LDB + c8), kg + off, in ? 16u : 0u);
      sm100::cp_async16(sm100::smem_addr(Qb + r * LDB + c8), qg + off, in ? 16u : 0u);
    }
  }
  {
    for (int idx = tid; idx < C * DK / 4; idx += kThreads) {
      const int r = idx / (DK / 4), c4 = (idx % (DK / 4)) * 4;
      const bool in = r < L;
      sm100::cp_async16(sm100::smem_addr(Gs + r * LDG + c4), a.g + ((long)(t0 + (in ? r : 0)) * a.HV + hv) * DK + c4,
                 in ? 16u : 0u);
    }
  }
  for (int r = tid; r < C; r += kThreads) {
    const bool in = r < L;
    sm100::cp_async4(sm100::smem_addr(Bs + r), a.beta + (long)(t0 + (in ? r : 0)) * a.HV + hv, in ? 4u : 0u);
  }
  for (int idx = tid; idx < C * LDC; idx += kThreads) Ts[idx] = 0.f;
  sm100::cp_async_wait_all();
  __syncthreads();
  bool positive = false;
  {
    for (int idx = tid; idx < C * DK; idx += kThreads) positive |= Gs[(idx / DK) * LDG + idx % DK] > 0.f;
  }
  if (__syncthreads_or(positive) && tid == 0) atomicOr(a.flags, kFlagPositiveGate);

  // ---- cumulative log-gates ----
  {
    for (int c = tid; c < DK; c += kThreads) {
      float run = 0.f;
      for (int r = 0; r < C; r++) {
        run += Gs[r * LDG + c];
        Gs[r * LDG + c] = run;
      }
    }
  }
  __syncthreads();

  // ---- A and Aqk ----
  {
    // Per 16-row block I with reference row o = 16 I:
    //   A[r][s]   = beta_r sum_c (k_rc e^{b_rc - b_oc}) (k_sc e^{b_oc - b_sc})
    //   Aqk[r][s] = scale  sum_c (q_rc e^{b_rc - b_oc}) (k_sc e^{b_oc - b_sc})
    // r in the block, s <= o + 15: the row factors are <= 1, the column factors
    // <= 1 for s <= o and at most e^{-(sum of the block's gates)} inside it.
    // Products on the tensor cores in split bf16: each factored operand is
    // written once as hi + lo bf16 planes (16 significant bits, the fp32
    // exponent range the factors need) and read back by ldmatrix.  When an
    // in-block factor could leave the fp32 range the CTA falls back to forming
    // every pairwise decay directly.
    constexpr int LDH = SM::LDH;
    __nv_bfloat16 *Xkh = reinterpret_cast<__nv_bfloat16 *>(smem + SM::kX);
    __nv_bfloat16 *Xkl = Xkh + 16 * LDH, *Xqh = Xkl + 16 * LDH, *Xql = Xqh + 16 * LDH;
    __nv_bfloat16 *Khh = Xql + 16 * LDH, *Khl = Khh + C * LDH;
    bool wide = false;
    for (int idx = tid; idx < C * DK; idx += kThreads) {
      const int s = idx / DK, c = idx % DK, o = s & ~15;
      wide |= fabsf(Gs[o * LDG + c] - Gs[s * LDG + c]) > 80.f;
    }
    const bool pairwise = __syncthreads_or(wide);
    if (!pairwise) {
      for (int I = 0; I < C / 16; I++) {
        const int o = 16 * I, ns = o + 16;  // columns s < ns
        // four channels at a time
        auto bf4 = [](const __nv_bfloat16 *p) {
          const uint2 u = *reinterpret_cast<const uint2 *>(p);
          const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
          const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
          return make_float4(lo.x, lo.y, hi.x, hi.y);
        };
        for (int idx = tid; idx < 16 * DK / 4; idx += kThreads) {
          const int r = idx / (DK / 4), c = (idx % (DK / 4)) * 4;
          const float4 b = *reinterpret_cast<const float4 *>(Gs + (o + r) * LDG + c);
          const float4 bo = *reinterpret_cast<const float4 *>(Gs + o * LDG + c);
          const float4 e = make_float4(__expf(b.x - bo.x), __expf(b.y - bo.y), __expf(b.z - bo.z), __expf(b.w - bo.w));
          const float4 kv = bf4(Kb + (o + r) * LDB + c), qv = bf4(Qb + (o + r) * LDB + c);
          uint2 h, l;
          split4(make_float4(kv.x * e.x, kv.y * e.y, kv.z * e.z, kv.w * e.w), h, l);
          *reinterpret_cast<uint2 *>(Xkh + r * LDH + c) = h;
          *reinterpret_cast<uint2 *>(Xkl + r * LDH + c) = l;
          split4(make_float4(qv.x * e.x, qv.y * e.y, qv.z * e.z, qv.w * e.w), h, l);
          *reinterpret_cast<uint2 *>(Xqh + r * LDH + c) = h;
          *reinterpret_cast<uint2 *>(Xql + r * LDH + c) = l;
        }
        for (int idx = tid; idx < ns * DK / 4; idx += kThreads) {
          const int r = idx / (DK / 4), c = (idx % (DK / 4)) * 4;
          const float4 b = *reinterpret_cast<const float4 *>(Gs + r * LDG + c);
          const float4 bo = *reinterpret_cast<const float4 *>(Gs + o * LDG + c);
          const float4 kv = bf4(Kb + r * LDB + c);
          uint2 h, l;
          split4(make_float4(kv.x * __expf(bo.x - b.x), kv.y * __expf(bo.y - b.y),
                             kv.z * __expf(bo.z - b.z), kv.w * __expf(bo.w - b.w)), h, l);
          *reinterpret_cast<uint2 *>(Khh + r * LDH + c) = h;
          *reinterpret_cast<uint2 *>(Khl + r * LDH + c) = l;
        }
        __syncthreads();
        // tiles of 8 columns: ns / 8 for A, as many for Aqk.  Per 16-deep step
        // the fragments come by ldmatrix from the hi / lo planes and three
        // bf16 products (hi hi, lo hi, hi lo) accumulate in fp32.
        const int ntile = ns / 8;
        const uint32_t a_row = (lane & 15) * LDH + (lane >> 4) * 8;       // A fragment row
        const uint32_t b_row = (lane & 7) * LDH + ((lane >> 3) & 1) * 8;  // B fragment row
        for (int tile = warp; tile < 2 * ntile; tile += kThreads / 32) {
          const bool isq = tile >= ntile;
          const int n0 = 8 * (isq ? tile - ntile : tile);
          const uint32_t sAh = sm100::smem_addr(isq ? Xqh : Xkh) + 2 * a_row;
          const uint32_t sAl = sm100::smem_addr(isq ? Xql : Xkl) + 2 * a_row;
          const uint32_t sBh = sm100::smem_addr(Khh + n0 * LDH) + 2 * b_row;
          const uint32_t sBl = sm100::smem_addr(Khl + n0 * LDH) + 2 * b_row;
          float acc[4] = {0.f, 0.f, 0.f, 0.f}, corr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
          for (int k0 = 0; k0 < DK; k0 += 16) {
            uint32_t ah[4], al[4], bh0, bh1, bl0, bl1;
            ldsm_x4(ah, sAh + 2 * k0);
            ldsm_x4(al, sAl + 2 * k0);
            ldsm_x2(bh0, bh1, sBh + 2 * k0);
            ldsm_x2(bl0, bl1, sBl + 2 * k0);
            mma16816(acc, ah, bh0, bh1);
            mma16816(corr, al, bh0, bh1);
            mma16816(corr, ah, bl0, bl1);
          }
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const int r = o + acc_row(e), sc = n0 + acc_col(0, e);
            const float v = acc[e] + corr[e];
            if (isq) Aqks[r * LDC + sc] = sc <= r ? a.scale * v : 0.f;
            else As[r * LDC + sc] = sc < r ? Bs[r] * v : 0.f;
          }
        }
        __syncthreads();
      }
    } else {
    constexpr int NPAIR = C * (C + 1) / 2;
    for (int p = warp; p < NPAIR; p += kThreads / 32) {
      int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
      while ((r + 1) * (r + 2) / 2 <= p) r++;
      while (r * (r + 1) / 2 > p) r--;
      const int s = p - r * (r + 1) / 2;
      float kk = 0.f, qk = 0.f;
      for (int c = lane; c < DK; c += 32) {
        const float d = __expf(Gs[r * LDG + c] - Gs[s * LDG + c]);
        const float ks = __bfloat162float(Kb[s * LDB + c]) * d;
        kk += __bfloat162float(Kb[r * LDB + c]) * ks;
        qk += __bfloat162float(Qb[r * LDB + c]) * ks;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        kk += __shfl_xor_sync(0xffffffffu, kk, off);
        qk += __shfl_xor_sync(0xffffffffu, qk, off);
      }
      if (lane == 0) {
        As[r * LDC + s] = s < r ? Bs[r] * kk : 0.f;
        Aqks[r * LDC + s] = a.scale * qk;
      }
    }
    }
    for (int idx = tid; idx < C * C; idx += kThreads) {
      const int r = idx / C, s = idx % C;
      if (s > r) { As[r * LDC + s] = 0.f; Aqks[r * LDC + s] = 0.f; }
    }
  }
  __syncthreads();

  // ---- T = (I + A)^-1 ----
  constexpr int NB = C / 16;
  if (tid < NB * 16) {
    // diagonal block I, column j: right-looking substitution
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
  __syncthreads();
  // block row I:  R = A[I, 0:I] T[0:I, 0:I],  T[I, 0:I] = -T_II R
  for (int I = 1; I < NB; I++) {
    const int w = 16 * I;  // width of the solved part
    for (int idx = tid; idx < 16 * w; idx += kThreads) {
      const int m = idx / w, j = idx % w;
      float acc = 0.f;
      for (int s = (j & ~15); s < w; s++) acc += As[(w + m) * LDC + s] * Ts[s * LDC + j];
      Rs[m * LDC + j] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < 16 * w; idx += kThreads) {
      const int m = idx / w, j = idx % w;
      float acc = 0.f;
      for (int p = 0; p <= m; p++) acc += Ts[(w + m) * LDC + w + p] * Rs[p * LDC + j];
      Ts[(w + m) * LDC + j] = -acc;
    }
    __syncthreads();
  }

  // ---- KDA: the scan's operands, published while b, K and Q are at hand:
  //      the gated fp16 image [K~ = k e^b; Q~ = scale q e^b] (128 rows, K-major,
  //      128-byte swizzle; rows past the tokens zero) and e^{b_last} ----
  {
    unsigned char *kqi = a.kq_images + ((size_t)slot * a.HV + hv) * kq_image_bytes(DK);
    constexpr int NCH = (DK / 64) * 128 * 8;  // 16-byte chunks of the image
    for (int idx = tid; idx < NCH; idx += kThreads) {
      const int p = idx >> 10, rr = (idx >> 3) & 127, phys = idx & 7;
      const int half = rr >> 6, r = rr & 63;
      const int c0 = p * 64 + ((phys ^ (rr & 7)) << 3);  // first channel of the chunk
      uint4 out = make_uint4(0, 0, 0, 0);
      if (r < L) {
        const __nv_bfloat16 *src = (half ? Qb : Kb) + r * LDB + c0;
        const float mul = half ? a.scale : 1.f;
        __half2 *h = reinterpret_cast<__half2 *>(&out);
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const float e0 = __expf(Gs[r * LDG + c0 + 2 * i]), e1 = __expf(Gs[r * LDG + c0 + 2 * i + 1]);
          h[i] = __floats2half2_rn(mul * __bfloat162float(src[2 * i]) * e0,
                                   mul * __bfloat162float(src[2 * i + 1]) * e1);
        }
      }
      *reinterpret_cast<uint4 *>(kqi + p * 16384 + rr * 128 + phys * 16) = out;
    }
    for (int c = tid; c < DK; c += kThreads)
      a.decays[((size_t)slot * a.HV + hv) * DK + c] = __expf(Gs[(C - 1) * LDG + c]);
    __syncthreads();  // the gates below are overwritten in place
  }
  // ---- KDA: Kt = k * exp(b_last - b) in place of the cumulative gates ----
  {
    for (int c = tid; c < DK; c += kThreads) {
      const float bl = Gs[(C - 1) * LDG + c];
      for (int r = 0; r < C; r++)
        Gs[r * LDG + c] = __bfloat162float(Kb[r * LDB + c]) * __expf(bl - Gs[r * LDG + c]);
    }
  }
  __syncthreads();  // Kt complete; every reader of the X planes is done
  // ---- fp16 operands of the image products, into the dead X region ----
  {
    unsigned char *opKt = smem + SM::kOpKt, *opT = smem + SM::kOpT, *opAqk = smem + SM::kOpAqk;
    // Kt: token row r, channels 8 at a time (two panels, the second zero when dk = 64)
    for (int idx = tid; idx < C * 16; idx += kThreads) {
      const int r = idx / 16, c8 = (idx % 16) * 8;
      uint4 pk = make_uint4(0, 0, 0, 0);
      if (c8 < DK) {
        __half2 *h = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
        for (int i = 0; i < 4; i++) h[i] = __floats2half2_rn(Gs[r * LDG + c8 + 2 * i], Gs[r * LDG + c8 + 2 * i + 1]);
      }
      *reinterpret_cast<uint4 *>(opKt + sm100::kmajor_off(r, c8, C)) = pk;
    }
    // T as the B operand (row j = T[.][j]) and Aqk as the A operand (row r =
    // Aqk[r][.]), 64 columns per row, zero beyond C
    for (int idx = tid; idx < 2 * C * 8; idx += kThreads) {
      const bool isT = idx < C * 8;
      const int row = (idx % (C * 8)) / 8, k8 = (idx % 8) * 8;
      uint4 pk = make_uint4(0, 0, 0, 0);
      if (k8 < C) {
        __half2 *h = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const int k = k8 + 2 * i;
          h[i] = isT ? __floats2half2_rn(Ts[k * LDC + row], Ts[(k + 1) * LDC + row])
                     : __floats2half2_rn(Aqks[row * LDC + k], Aqks[row * LDC + k + 1]);
        }
      }
      *reinterpret_cast<uint4 *>((isT ? opT : opAqk) + sm100::kmajor_off(row, k8, isT ? C : 128)) = pk;
    }
    // the output image (Q and A are dead now) starts at zero
    for (int idx = tid; idx < kPrepImageBytes / 16; idx += kThreads)
      reinterpret_cast<uint4 *>(img)[idx] = make_uint4(0, 0, 0, 0);
  }
  sm100::fence_proxy_async();
  sm100::fence_before_sync();
  __syncthreads();
  sm100::fence_after_sync();
  const uint32_t tmem = *tslot;
  // ---- P1 = Kt^T T (M = dk rows, N = C, K = C) and Aqk T (rows < C) on
  //      the tensor cores, fp16 operands, fp32 accumulation ----
  if (tid == 0) {
    const uint32_t sKt = sm100::smem_addr(smem + SM::kOpKt), sT = sm100::smem_addr(smem + SM::kOpT);
    const uint32_t sAqk = sm100::smem_addr(smem + SM::kOpAqk);
    constexpr uint32_t idP = sm100::idesc_f16(128, C, 1, 0);  // Kt read MN-major
    constexpr uint32_t idQ = sm100::idesc_f16(128, C, 0, 0);
#pragma unroll
    for (int k0 = 0; k0 < C; k0 += 16) {
      const uint64_t bd = sm100::make_desc(sT + k0 * 2, 16, 1024);
      sm100::mma_f16(tmem, sm100::make_desc(sKt + k0 * 128, C * 128, 1024), bd, idP, k0 > 0 ? 1u : 0u);
      sm100::mma_f16(tmem + 64, sm100::make_desc(sAqk + k0 * 2, 16, 1024), bd, idQ, k0 > 0 ? 1u : 0u);
    }
    sm100::mma_commit(bar_mma);
  }
  sm100::mbar_wait(bar_mma, 0, abort_flag);
  sm100::fence_after_sync();
  // ---- read back: lane t holds row t of P1 (t < dk) and of Aqk T (t < C) ----
  {
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    auto put_row = [&](int row, uint32_t taddr) {
#pragma unroll
      for (int h = 0; h < C / 32; h++) {
        uint32_t v[32];
        sm100::tmem_ld32_nowait(taddr + 32 * h, v);
        sm100::tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < 4; ch++) {
          uint4 pk;
          __half2 *hh = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
          for (int i = 0; i < 4; i++)
            hh[i] = __floats2half2_rn(__uint_as_float(v[ch * 8 + 2 * i]), __uint_as_float(v[ch * 8 + 2 * i + 1]));
          *reinterpret_cast<uint4 *>(img + sm100::kmajor_off(row, 32 * h + ch * 8, kPrepImageRows)) = pk;
        }
      }
    };
    if (tid < DK) put_row(tid, tmem + lane_base);
    if (tid < C) put_row(kPrepImageRows - 64 + tid, tmem + lane_base + 64);
  }
  sm100::fence_proxy_async();
  sm100::fence_before_sync();
  __syncthreads();
  sm100::fence_after_sync();

  // ---- image -> workspace, one bulk copy ----
  if (tid == 0) {
    unsigned char *dst = reinterpret_cast<unsigned char *>(a.tiles) + ((size_t)slot * a.HV + hv) * kPrepImageBytes;
    sm100::bulk_s2g(dst, sm100::smem_addr(img), kPrepImageBytes);
    sm100::bulk_commit();
    sm100::bulk_wait_read_all();
    if (*abort_flag) atomicOr(a.flags, kFlagTimeout);
  }
  __syncthreads();
  if (warp == 0) sm100::tmem_dealloc(tmem, kTmemCols);
}

template <int C, int DK>
cudaError_t launch_one(const PrepArgs &a, cudaStream_t stream) {
  using SM = PrepTcSmem<C, DK>;
  auto kern = gdn_prep_tc_kernel<C, DK>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (err != cudaSuccess) return err;
  kern<<<dim3(a.n_slots, a.HV), kThreads, SM::kBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_tc(const PrepArgs &a, int chunk, int dk, int gate, cudaStream_t stream) {
  if (!gate) return cudaErrorInvalidValue;  // the scalar gate runs gdn_prep_tmem.cu
  if (chunk == 64 && dk == 128) return launch_one<64, 128>(a, stream);
  if (chunk == 64 && dk == 64) return launch_one<64, 64>(a, stream);
  if (chunk == 32 && dk == 128) return launch_one<32, 128>(a, stream);
  if (chunk == 32 && dk == 64) return launch_one<32, 64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
