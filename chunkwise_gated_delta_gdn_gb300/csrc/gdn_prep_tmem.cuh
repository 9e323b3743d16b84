// gdn_prep_tmem.cuh -- the chunk-prep computation of the bf16 scalar-gate
// (GDN) path on the 5th-generation tensor cores, as a device function over one
// (chunk slot, q/k head) unit run by one warpgroup.  gdn_prep_tmem.cu launches
// it as one CTA per unit; the lockstep kernel (gdn_lockstep.cu) runs it in
// persistent warpgroups beside the scan.
//
// Per (chunk slot, q/k head), one warpgroup (128 threads) takes the group's
// value heads in turn, holding 128 tensor-memory columns and about 75 KB of
// shared memory.  The group shares the key/query tile and the
// next chunk's key tile: they arrive once by TMA (bf16, 128-byte swizzle), are
// converted to fp16 in place, published for the scan kernel as its
// [K_next; Q] operand image, and feed one Gram product for all value heads:
//   G  = [K; Q] K^T          M = 128 (keys then queries), N = C, K = dk
// Then, for each value head in turn (gates and beta differ per head):
//   A    = strict-lower(beta_r G_rs exp(b_r - b_s)), Aqk = lower(scale P_rs
//          exp(b_r - b_s)) straight from its tensor-memory lanes; inside a
//          32-row block the decay is one exp2 per entry, across blocks it is
//          exp(b_r - b_o) exp(b_o - b_s) with o the block's first row (both
//          factors <= 1 for non-positive gates: nothing overflows)
//   T    = (I + A)^-1 blocked as in ROCm/rocm-libraries PR #11223 ("Levers"
//          3): each 16 x 16 diagonal block by fp32 forward substitution in
//          registers (one lane per column), then the 32 x 32 and 64 x 64 levels
//          T10 = -T11 (A10 T00) as one-pass fp16 mma.sync products with fp32
//          accumulation (T itself enters the later products as fp16 anyway)
//   P1   = K^T (D T)         the key tile read MN-major, D = diag(exp(b_last - b_s))
//   AqkT = Aqk T
//   E    = K_next P1         (fp16 P1 as the B operand; zero for the last chunk
//                             of a sequence)
// and writes them, each rounded once to fp16, as the 32 KB operand image of the
// lookahead scan kernel (rows 0..127 = P1, 128..191 = E, 192..255 = AqkT;
// K-major, 128-byte swizzle), staged in shared memory over buffers that are
// dead by then and stored with three bulk copies.  The three products take
// turns in one 64-column tensor-memory buffer.  The staged P1 rows double as
// E's B operand: a K-major image of P1's dk rows is the MN-major layout of P1
// read as a dk x C operand.  E lets the scan form
// the next chunk's K S from this chunk's Y without waiting for the state:
//   K_next S_next = exp(b_last) K_next S + E Y.
#pragma once

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

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int C>
struct PrepTmemSmem {
  static constexpr int LDT = 68;                    // fp32 row stride of A^T / T^T
  // [K; Q; K_next] of each 64-column panel of the key/query dimension,
  // K-major, 192 rows x 128 bytes; two panels (room for dk = 128), PSTR apart
  static constexpr int PANEL = 192 * 128;
  static constexpr int PSTR = PANEL + 1024;
  static constexpr int kKQ = 0;
  // Once both Gram products have read the query and next-key rows and the
  // [K_next; Q] image has been stored, those rows hold the per-head buffers:
  //   X2  panel 0's rows 64..191 and the 1 KB after them: A^T, then T^T, in
  //       fp32 (row stride LDT), then the fp16 T and D T images (8 KB each),
  //       then the staged Aqk T rows (over T), then the staged P1 rows
  //   AG  panel 1's rows 64..191: the fp16 Aqk image (later the staged E
  //       rows), then the image of Gn = K_next K^T; read together as one
  //       128-row operand
  static constexpr int kX2 = 64 * 128;
  static constexpr int kAG = PSTR + 64 * 128;
  static constexpr int kGn = kAG + 64 * 128;
  static constexpr int kW = PSTR + PANEL;           // W scratch of the solve
  static constexpr int kG = kW + 4 * 32 * 9 * 4;    // cumulative gates (log2 units)
  static constexpr int kBeta = kG + C * 4;
  static constexpr int kDec = kBeta + C * 4;
  static constexpr int kWf = kDec + C * 4;          // cross-block decay factors (32)
  static constexpr int kBar = kWf + 32 * 4;         // tma, gram, mma
  static constexpr int kMisc = kBar + 3 * 8;
  // a CTA running one unit at a time: the layout plus 1 KB of alignment
  // slack; a CTA of several warpgroups gives each a slice of kSlice bytes (a
  // 1 KB multiple) and adds the slack once.  The first word at kMisc is left
  // to the caller (its tensor-memory address slot).
  static constexpr int kBytes = kMisc + 32 + 1024;
  static constexpr int kSlice = (kMisc + 32 + 1023) / 1024 * 1024;
  static_assert(C * LDT * 4 <= PSTR - kX2, "A^T in X2");
  static_assert(kBar % 8 == 0, "mbarrier alignment");
  // four CTAs per SM: 228 KB of shared memory, 1 KB of it reserved per CTA
  static_assert(4 * (kBytes + 1024) <= 233472, "four CTAs per SM");
};

// Completions seen so far of the three mbarriers of a warpgroup's slice (the
// TMA tiles, the Gram product, the later products): a warpgroup initialises
// its barriers once and carries these counts from one unit to the next.
struct PrepPhases {
  uint32_t tma = 0, gram = 0, mma = 0;
};

// Initialise the mbarriers of a slice (one thread; the warpgroup synchronises
// before the first unit).
template <int C>
__device__ __forceinline__ void prep_tmem_init_barriers(unsigned char *sm) {
  using SM = PrepTmemSmem<C>;
  const uint32_t bar0 = smem_addr(sm + SM::kBar);
  mbar_init(bar0, 1);       // TMA tiles
  mbar_init(bar0 + 8, 1);   // Gram product
  mbar_init(bar0 + 16, 1);  // P1, Aqk T, E products
  mbar_fence_init();
}

// One (chunk slot, q/k head) unit, run by one warpgroup.
//   sm      its shared memory (PrepTmemSmem<C>::kSlice bytes, 1 KB aligned)
//   tmem    the first of its 128 tensor-memory columns (allocated by the caller)
//   tid     the thread's index in the warpgroup (0..127); the warpgroup's
//           warps are four consecutive warps starting at a multiple of four
//   bar_id  the named barrier of the warpgroup
//   ready   when given, the unit's operand images are complete in global
//           memory before ready[slot * H + hq] is set to 1 (release, gpu scope)
//   ph      the warpgroup's barrier completion counts (prep_tmem_init_barriers
//           ran once before its first unit)
template <int C, int DK>
__device__ __forceinline__ void prep_tmem_unit(const PrepArgs &a, const ScanMaps &maps, int slot,
                                               int hq, unsigned char *sm, uint32_t tmem,
                                               int tid, int bar_id, int *ready, PrepPhases &ph) {
  using SM = PrepTmemSmem<C>;
  constexpr int LDT = SM::LDT;
  constexpr int NT = 128;
  unsigned char *kq = sm + SM::kKQ;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM::kBar);
  const uint32_t bar_tma = smem_addr(bars), bar_gram = smem_addr(bars + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SM::kMisc + 4);
  int *meta = reinterpret_cast<int *>(sm + SM::kMisc + 8);

  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;

  // ---- slot -> (sequence, chunk) ----
  named_bar(bar_id, 128);  // a persistent warpgroup: the last unit's reads of meta are done
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
    // tokens of the sequence's next chunk (0 for its last chunk)
    meta[3] = (valid && t0 + C < end) ? (int)min((long)C, (long)end - t0 - C) : 0;
    *abort_flag = 0;
  }
  named_bar(bar_id, 128);
  if (!meta[2]) return;  // unused slot: the scan never reads it
  const int t0 = meta[0], L = meta[1], Ln = meta[3];

  // Gram (C columns) at 0; Gn, then Aqk T, E and P1 in turn, at 64
  if (C < 64) {  // zero the rows no TMA box covers
    for (int i = tid; i < 2 * SM::PANEL / 16; i += NT) {
      const int p = i / (SM::PANEL / 16), w = i % (SM::PANEL / 16);
      if (((w / 8) & 63) >= C)
        *reinterpret_cast<uint4 *>(kq + p * SM::PSTR + w * 16) = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_tma, (Ln > 0 ? 3 : 2) * C * DK * 2);
#pragma unroll
    for (int p = 0; p < DK / 64; p++) {
      tma_load_3d(smem_addr(kq + p * SM::PSTR), &maps.k, p * 64, hq, t0, bar_tma);
      tma_load_3d(smem_addr(kq + p * SM::PSTR + 64 * 128), &maps.q, p * 64, hq, t0, bar_tma);
      if (Ln > 0) tma_load_3d(smem_addr(kq + p * SM::PSTR + 128 * 128), &maps.k, p * 64, hq, t0 + C, bar_tma);
    }
  }
  // value head j's raw gates and beta by cp.async (zeros past the chunk's
  // tokens) into the end-of-chunk decay and beta arrays, which are free from
  // the previous head's T images to this head's gate phase: the first head's
  // land while the tiles do, each later head's while the previous head's
  // products run.  Thread t copies and later reads only its own row.
  const int t = tid;
  const int G = a.HV / a.H;
  float *raw_g = reinterpret_cast<float *>(sm + SM::kDec);
  float *raw_b = reinterpret_cast<float *>(sm + SM::kBeta);
  auto fetch = [&](int j) {
    if (t < C && j < G) {
      const bool in = t < L;
      const long row = (long)(t0 + (in ? t : 0)) * a.HV + hq * G + j;
      cp_async4(smem_addr(raw_g + t), a.g + row, in ? 4u : 0u);
      cp_async4(smem_addr(raw_b + t), a.beta + row, in ? 4u : 0u);
    }
  };
  fetch(0);
  mbar_wait(bar_tma, ph.tma++ & 1, abort_flag);
  // bf16 -> fp16 in place; rows beyond each tile's tokens -> 0.  Six 16-byte
  // chunks per thread in flight at a time (the loop is shared-memory latency
  // bound otherwise).
  {
    constexpr int CH = (DK / 64) * 3 * C * 8;
    constexpr int PER = CH / NT, UNR = 6;
    static_assert(CH % NT == 0 && PER % UNR == 0, "conversion tiling");
#pragma unroll 1
    for (int b0 = 0; b0 < PER; b0 += UNR) {
      uint4 v[UNR];
      uint4 *ptr[UNR];
      bool keep[UNR];
#pragma unroll
      for (int u = 0; u < UNR; u++) {
        const int idx = tid + (b0 + u) * NT;
        const int p = idx / (3 * C * 8), rem = idx % (3 * C * 8);
        const int third = rem / (C * 8), r = (rem / 8) % C, chunk = rem % 8;
        ptr[u] = reinterpret_cast<uint4 *>(kq + p * SM::PSTR + (third * 64 + r) * 128 + chunk * 16);
        keep[u] = r < (third == 2 ? Ln : L);
        v[u] = keep[u] ? *ptr[u] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < UNR; u++) {
        uint4 out = make_uint4(0, 0, 0, 0);
        if (keep[u]) {
          const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&v[u]);
          __half2 *h = reinterpret_cast<__half2 *>(&out);
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const float2 f = __bfloat1622float2(b[i]);
            h[i] = __floats2half2_rn(f.x, f.y);
          }
        }
        *ptr[u] = out;
      }
    }
  }
  fence_proxy_async();
  fence_before_sync();
  named_bar(bar_id, 128);
  fence_after_sync();
  // ---- G = [K; Q] K^T (columns [0, C)) and [Q; K_next] K^T (columns
  //      [64, 64 + C)), whose lanes 64.. hold Gn = K_next K^T ----
  const uint32_t tX = tmem + 64;  // Gn, then Aqk T, E and P1 in turn
  if (tid == 0) {
    const uint32_t sKQ = smem_addr(kq);
    constexpr uint32_t id = idesc_f16(128, C, 0, 0);
#pragma unroll
    for (int k0 = 0; k0 < DK; k0 += 16) {
      const uint32_t base = sKQ + (k0 >> 6) * SM::PSTR + (k0 & 63) * 2;
      const uint64_t d = make_desc(base, 16, 1024);  // [K; Q], and its key rows as B
      mma_f16(tmem, d, d, id, k0 > 0 ? 1u : 0u);
      mma_f16(tX, make_desc(base + 64 * 128, 16, 1024), d, id, k0 > 0 ? 1u : 0u);
    }
    mma_commit(bar_gram);
  }
  // publish [K_next; Q] (rows 128.. and 64.. of each panel) while the Gram
  // runs: bulk stores, completed before the CTA ends
  if (tid == 0) {
    unsigned char *dst = a.kq_images + ((size_t)slot * a.H + hq) * kq_image_bytes(DK);
#pragma unroll
    for (int p = 0; p < DK / 64; p++) {
      bulk_s2g(dst + p * 16384, smem_addr(kq + p * SM::PSTR + 16384), 8192);
      bulk_s2g(dst + p * 16384 + 8192, smem_addr(kq + p * SM::PSTR + 8192), 8192);
    }
    bulk_commit();
  }

  // this lane's row at `taddr` -> row `row` of a 64-column K-major fp16
  // image at `dst` (zeros when !have)
  auto put_row = [&](unsigned char *dst, int row, uint32_t taddr, bool have) {
#pragma unroll
    for (int h = 0; h < 2; h++) {  // 32 columns at a time
      uint32_t v[32];
      if (have && 32 * h < C) {
        tmem_ld32_nowait(taddr + 32 * h, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; i++) v[i] = 0u;
      }
#pragma unroll
      for (int ch = 0; ch < 4; ch++) {
        uint4 pk;
        __half2 *hh = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
        for (int i = 0; i < 4; i++)
          hh[i] = __floats2half2_rn(__uint_as_float(v[ch * 8 + 2 * i]), __uint_as_float(v[ch * 8 + 2 * i + 1]));
        *reinterpret_cast<uint4 *>(dst + kmajor_off(row, 32 * h + ch * 8, 64)) = pk;
      }
    }
  };

  // ---- per value head ----
  float *As = reinterpret_cast<float *>(sm + SM::kX2);
  float *Rs = reinterpret_cast<float *>(sm + SM::kW);  // W scratch of the solve
  float *Gs = reinterpret_cast<float *>(sm + SM::kG);
  float *Bs = reinterpret_cast<float *>(sm + SM::kBeta);
  float *Ds = reinterpret_cast<float *>(sm + SM::kDec);
  const uint32_t bar_mma = bar_tma + 16;
  const int wlane0 = (warp & 3) * 32;  // first tensor-memory lane of this warp
  const uint32_t sKQ = smem_addr(kq), sX2 = smem_addr(sm + SM::kX2), sAG = smem_addr(sm + SM::kAG);
  bool first = true;
  float *Wf = reinterpret_cast<float *>(sm + SM::kWf);  // exp2(b_32 - b_s), s < 32
  for (int j = 0; j < G; j++) {
    const int hv = hq * G + j;
    // the previous head's image stores must have read the buffers reused below
    if (j > 0) {
      if (t == 0) bulk_wait_read_all();
      named_bar(bar_id, 128);
    }
    // gates (log2 units), beta, cumulative gates, end-of-chunk decays
    cp_async_wait_all();  // this head's raw gates (in Ds) and beta (in Bs)
    const float gv = t < C ? raw_g[t] : 0.f;
    bool positive = false;
    if (t < C) {
      positive = gv > 0.f;
      Gs[t] = gv * kLog2e;
    }
    if (__any_sync(0xffffffffu, positive) && lane == 0) atomicOr(a.flags, kFlagPositiveGate);
    named_bar(bar_id, 128);
    if ((warp & 3) == 0) {
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
      if (lane < C) { Gs[lane] = x0; Ds[lane] = ex2(blast - x0); }
      if (lane + 32 < C) { Gs[lane + 32] = x1; Ds[lane + 32] = ex2(blast - x1); }
      if (C > 32) Wf[lane] = ex2(__shfl_sync(0xffffffffu, x1, 0) - x0);
    }
    if (first) {
      // the Gram products are done, and the [K_next; Q] image store has read
      // the rows that the per-head buffers reuse; Gn's rows -> its image
      mbar_wait(bar_gram, ph.gram++ & 1, abort_flag);
      if (t == 0) bulk_wait_read_all();
      named_bar(bar_id, 128);
      fence_after_sync();
      if (t >= 64) put_row(sm + SM::kGn, t - 64, tX + lane_base, wlane0 - 64 < C);
      first = false;
    }
    named_bar(bar_id, 128);

    // ---- A (key lanes) and Aqk (query lanes) from the shared Gram ----
    // decay of column s for row r in 32-row block o: direct inside the block,
    // factored (ur * Wf[s]) for the earlier block.  A is stored transposed
    // (As[s * LDT + r] = A[r][s]): the solve reads its columns as rows.
    if (wlane0 < C) {
      const int r = t, o = wlane0;
      const float br = Gs[r], beta = Bs[r];
      const float bu = o > 0 ? beta * ex2(br - Gs[o]) : 0.f;
#pragma unroll
      for (int h = 0; h < C / 32; h++) {
        if (32 * h > o) {  // s > r throughout
#pragma unroll
          for (int i = 0; i < 32; i++) As[(32 * h + i) * LDT + r] = 0.f;
          continue;
        }
        uint32_t g[32];
        tmem_ld32_nowait(tmem + lane_base + 32 * h, g);
        tmem_wait_ld();
        // the block's 32 column factors (cross-block factors or cumulative
        // gates), four at a time
        float fv[32];
        {
          const float *src = 32 * h < o ? Wf : Gs + 32 * h;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 f4 = *reinterpret_cast<const float4 *>(src + i);
            fv[i] = f4.x; fv[i + 1] = f4.y; fv[i + 2] = f4.z; fv[i + 3] = f4.w;
          }
        }
        if (32 * h < o) {
#pragma unroll
          for (int i = 0; i < 32; i++) As[(32 * h + i) * LDT + r] = bu * __uint_as_float(g[i]) * fv[i];
        } else {
#pragma unroll
          for (int i = 0; i < 32; i++) {
            const int s = 32 * h + i;
            As[s * LDT + r] = s < r ? beta * __uint_as_float(g[i]) * ex2(br - fv[i]) : 0.f;
          }
        }
      }
    } else if (wlane0 >= 64 && wlane0 - 64 < C) {
      const int r = t - 64, o = wlane0 - 64;
      const float br = Gs[r];
      const float su = o > 0 ? a.scale * ex2(br - Gs[o]) : 0.f;
      unsigned char *aq = sm + SM::kAG;
#pragma unroll
      for (int h = 0; h < C / 32; h++) {
        if (32 * h > o) {  // s > r throughout: a zero block of Aqk
#pragma unroll
          for (int ch = 0; ch < 4; ch++)
            *reinterpret_cast<uint4 *>(aq + kmajor_off(r, 32 * h + ch * 8, 64)) = make_uint4(0, 0, 0, 0);
          continue;
        }
        uint32_t g[32];
        tmem_ld32_nowait(tmem + lane_base + 32 * h, g);
        tmem_wait_ld();
        float fv[32];
        {
          const float *src = 32 * h < o ? Wf : Gs + 32 * h;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 f4 = *reinterpret_cast<const float4 *>(src + i);
            fv[i] = f4.x; fv[i + 1] = f4.y; fv[i + 2] = f4.z; fv[i + 3] = f4.w;
          }
        }
#pragma unroll
        for (int ch = 0; ch < 4; ch++) {
          uint4 pk;
          __half2 *ph = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const int s = 32 * h + ch * 8 + 2 * i;
            const int ii = ch * 8 + 2 * i;
            float v0, v1;
            if (32 * h < o) {
              v0 = su * __uint_as_float(g[ii]) * fv[ii];
              v1 = su * __uint_as_float(g[ii + 1]) * fv[ii + 1];
            } else {
              v0 = s <= r ? a.scale * __uint_as_float(g[ii]) * ex2(br - fv[ii]) : 0.f;
              v1 = s + 1 <= r ? a.scale * __uint_as_float(g[ii + 1]) * ex2(br - fv[ii + 1]) : 0.f;
            }
            ph[i] = __floats2half2_rn(v0, v1);
          }
          *reinterpret_cast<uint4 *>(aq + kmajor_off(r, 32 * h + ch * 8, 64)) = pk;
        }
      }
    }
    fence_before_sync();
    named_bar(bar_id, 128);

    // ---- T = (I + A)^-1, transposed in place: As[j * LDT + r] = T[r][j] ----
    // (1) 16 x 16 diagonal blocks: warp w, lanes 0..15 = columns, rows in
    //     registers, forward substitution in fp32
    {
      const int wq = warp & 3;
      if (wq < C / 16 && lane < 16) {
        const int o = 16 * wq;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; r++) x[r] = r == lane ? 1.f : 0.f;
#pragma unroll
        for (int s2 = 0; s2 < 15; s2++) {
          const float xs = x[s2];
          const float *col = As + (o + s2) * LDT + o;  // A[o + r][o + s2], r = 0..15
#pragma unroll
          for (int m = (s2 + 1) / 4; m < 4; m++) {
            const float4 a4 = *reinterpret_cast<const float4 *>(col + 4 * m);
            if (4 * m + 0 > s2) x[4 * m + 0] = fmaf(-a4.x, xs, x[4 * m + 0]);
            if (4 * m + 1 > s2) x[4 * m + 1] = fmaf(-a4.y, xs, x[4 * m + 1]);
            if (4 * m + 2 > s2) x[4 * m + 2] = fmaf(-a4.z, xs, x[4 * m + 2]);
            if (4 * m + 3 > s2) x[4 * m + 3] = fmaf(-a4.w, xs, x[4 * m + 3]);
          }
        }
        __syncwarp(0x0000ffffu);
        float *row = As + (o + lane) * LDT + o;  // T[o + r][o + lane]
#pragma unroll
        for (int m = 0; m < 4; m++)
          *reinterpret_cast<float4 *>(row + 4 * m) = make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
      }
      named_bar(bar_id, 128);
      // (2) 32 x 32 blocks from their 16 x 16 halves: T10 = -T11 (A10 T00),
      //     one warp per (32-block, 8-column tile); one-pass fp16 tensor-core
      //     products with fp32 accumulation, W staged in the warp's rows of Rs
      const int gq = lane >> 2, tq = lane & 3;
      const bool act2 = wq < 2 * (C / 32);
      const int ob = 32 * (wq >> 1), n2 = 8 * (wq & 1);
      float *Wt2 = Rs + wq * 16 * 9;  // this warp's 16 x 8 W tile, row stride 9
      if (act2) {
        float w[4] = {0.f, 0.f, 0.f, 0.f};
        warp_mma_f16(w, 0, [&](int m, int k) { return As[(ob + k) * LDT + ob + 16 + m]; },
                     [&](int k, int n) { return As[(ob + n2 + n) * LDT + ob + k]; });
        Wt2[gq * 9 + 2 * tq] = w[0]; Wt2[gq * 9 + 2 * tq + 1] = w[1];
        Wt2[(gq + 8) * 9 + 2 * tq] = w[2]; Wt2[(gq + 8) * 9 + 2 * tq + 1] = w[3];
      }
      named_bar(bar_id, 128);  // both warps of a block have read A10 before T10 overwrites it
      if (act2) {
        float u[4] = {0.f, 0.f, 0.f, 0.f};
        warp_mma_f16(u, 0, [&](int m, int k) { return As[(ob + 16 + k) * LDT + ob + 16 + m]; },
                     [&](int k, int n) { return Wt2[k * 9 + n]; });
        // T10[r][c] -> As[(ob + n2 + c) LDT + ob + 16 + r], over A10^T
        As[(ob + n2 + 2 * tq) * LDT + ob + 16 + gq] = -u[0];
        As[(ob + n2 + 2 * tq + 1) * LDT + ob + 16 + gq] = -u[1];
        As[(ob + n2 + 2 * tq) * LDT + ob + 24 + gq] = -u[2];
        As[(ob + n2 + 2 * tq + 1) * LDT + ob + 24 + gq] = -u[3];
      }
      named_bar(bar_id, 128);
      if constexpr (C == 64) {
        // (3) the 64 x 64 inverse from its 32 x 32 halves: T10 = -T11 (A10 T00),
        //     warp w owns columns 8w .. 8w+7 of W and of T10
        const int n0 = 8 * wq;
        float w[2][4] = {};
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 16)
#pragma unroll
          for (int mt = 0; mt < 2; mt++)
            warp_mma_f16(w[mt], k0, [&](int m, int k) { return As[k * LDT + 32 + 16 * mt + m]; },
                         [&](int k, int n) { return As[(n0 + n) * LDT + k]; });
        float *Wt = Rs + wq * 32 * 9;  // this warp's 32 x 8 W tile, row stride 9
#pragma unroll
        for (int mt = 0; mt < 2; mt++) {
          Wt[(16 * mt + gq) * 9 + 2 * tq] = w[mt][0]; Wt[(16 * mt + gq) * 9 + 2 * tq + 1] = w[mt][1];
          Wt[(16 * mt + gq + 8) * 9 + 2 * tq] = w[mt][2]; Wt[(16 * mt + gq + 8) * 9 + 2 * tq + 1] = w[mt][3];
        }
        named_bar(bar_id, 128);  // every warp has read A10 before T10 overwrites it
        float u[2][4] = {};
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 16)
#pragma unroll
          for (int mt = 0; mt < 2; mt++)
            if (k0 < 16 * (mt + 1))  // T11 lower triangular
              warp_mma_f16(u[mt], k0, [&](int m, int k) { return As[(32 + k) * LDT + 32 + 16 * mt + m]; },
                           [&](int k, int n) { return Wt[k * 9 + n]; });
#pragma unroll
        for (int mt = 0; mt < 2; mt++) {
          As[(n0 + 2 * tq) * LDT + 32 + 16 * mt + gq] = -u[mt][0];
          As[(n0 + 2 * tq + 1) * LDT + 32 + 16 * mt + gq] = -u[mt][1];
          As[(n0 + 2 * tq) * LDT + 40 + 16 * mt + gq] = -u[mt][2];
          As[(n0 + 2 * tq + 1) * LDT + 40 + 16 * mt + gq] = -u[mt][3];
        }
        named_bar(bar_id, 128);
      }
    }

    // ---- fp16 images of T and D T as K-major B operands (row j = T[.][j]),
    //      over T^T's own space: every thread reads its 16-byte chunks, then
    //      all write ----
    {
      constexpr int NU = C * (C / 8) / NT;
      static_assert(C * (C / 8) % NT == 0, "image build tiling");
      uint4 pt[NU], pd[NU];
#pragma unroll
      for (int u = 0; u < NU; u++) {
        const int task = t + u * NT, jj = task % C, ch = task / C;
        const float *trow = As + jj * LDT;
        const float4 t0v = *reinterpret_cast<const float4 *>(trow + ch * 8);
        const float4 t1v = *reinterpret_cast<const float4 *>(trow + ch * 8 + 4);
        const float4 d0 = *reinterpret_cast<const float4 *>(Ds + ch * 8);
        const float4 d1 = *reinterpret_cast<const float4 *>(Ds + ch * 8 + 4);
        __half2 *ht = reinterpret_cast<__half2 *>(&pt[u]);
        __half2 *hd = reinterpret_cast<__half2 *>(&pd[u]);
        ht[0] = __floats2half2_rn(t0v.x, t0v.y); ht[1] = __floats2half2_rn(t0v.z, t0v.w);
        ht[2] = __floats2half2_rn(t1v.x, t1v.y); ht[3] = __floats2half2_rn(t1v.z, t1v.w);
        hd[0] = __floats2half2_rn(d0.x * t0v.x, d0.y * t0v.y); hd[1] = __floats2half2_rn(d0.z * t0v.z, d0.w * t0v.w);
        hd[2] = __floats2half2_rn(d1.x * t1v.x, d1.y * t1v.y); hd[3] = __floats2half2_rn(d1.z * t1v.z, d1.w * t1v.w);
      }
      named_bar(bar_id, 128);
#pragma unroll
      for (int u = 0; u < NU; u++) {
        const int task = t + u * NT, jj = task % C, ch = task / C;
        *reinterpret_cast<uint4 *>(sm + SM::kX2 + kmajor_off(jj, ch * 8, 64)) = pt[u];
        *reinterpret_cast<uint4 *>(sm + SM::kX2 + 8192 + kmajor_off(jj, ch * 8, 64)) = pd[u];
      }
    }
    fence_proxy_async();
    fence_before_sync();
    named_bar(bar_id, 128);
    fence_after_sync();
    // the decays and beta of this head are consumed: the next head's gates
    fetch(j + 1);

    // The image of this (chunk, value head): rows 0..127 = P1, 128..191 = E,
    // 192..255 = Aqk T.  [Aqk; Gn] is the A operand of both Aqk T (output
    // rows 0..63) and E = Gn (D T) (output rows 64..127).
    unsigned char *dst = reinterpret_cast<unsigned char *>(a.tiles) + ((size_t)slot * a.HV + hv) * kLaImageBytes;
    constexpr uint32_t idK = idesc_f16(128, C, 0, 0);
    // ---- Aqk T, staged over the T image ----
    if (t == 0) {
#pragma unroll
      for (int k0 = 0; k0 < C; k0 += 16)
        mma_f16(tX, make_desc(sAG + k0 * 2, 16, 1024), make_desc(sX2 + k0 * 2, 16, 1024), idK,
                k0 > 0 ? 1u : 0u);
      mma_commit(bar_mma);
    }
    mbar_wait(bar_mma, ph.mma++ & 1, abort_flag);
    fence_after_sync();
    if (t < 64) put_row(sm + SM::kX2, t, tX + lane_base, wlane0 < C);
    fence_proxy_async();
    fence_before_sync();
    named_bar(bar_id, 128);
    fence_after_sync();
    // ---- E = Gn (D T), staged over the Aqk image (zero for the last chunk
    //      of a sequence) ----
    if (t == 0) {
      bulk_s2g(dst + 192 * 128, sX2, 64 * 128);
      bulk_commit();
      if (Ln > 0) {
#pragma unroll
        for (int k0 = 0; k0 < C; k0 += 16)
          mma_f16(tX, make_desc(sAG + k0 * 2, 16, 1024), make_desc(sX2 + 8192 + k0 * 2, 16, 1024),
                  idK, k0 > 0 ? 1u : 0u);
        mma_commit(bar_mma);
      }
    }
    if (Ln > 0) {
      mbar_wait(bar_mma, ph.mma++ & 1, abort_flag);
      fence_after_sync();
    }
    if (t >= 64) put_row(sm + SM::kAG, t - 64, tX + lane_base, Ln > 0 && wlane0 - 64 < C);
    fence_proxy_async();
    fence_before_sync();
    named_bar(bar_id, 128);
    fence_after_sync();
    // ---- P1 = K^T (D T), the key tile read MN-major, staged over X2 ----
    if (t == 0) {
      bulk_s2g(dst + 128 * 128, sAG, 64 * 128);
      bulk_commit();
      constexpr uint32_t idP = idesc_f16(128, C, 1, 0);
#pragma unroll
      for (int k0 = 0; k0 < C; k0 += 16)
        mma_f16(tX, make_desc(sKQ + k0 * 128, SM::PSTR, 1024), make_desc(sX2 + 8192 + k0 * 2, 16, 1024),
                idP, k0 > 0 ? 1u : 0u);
      mma_commit(bar_mma);
    }
    mbar_wait(bar_mma, ph.mma++ & 1, abort_flag);
    if (t == 0) bulk_wait_read_1();  // the staged Aqk T rows have been read
    fence_before_sync();
    named_bar(bar_id, 128);
    fence_after_sync();
    put_row(sm + SM::kX2, t, tX + lane_base, wlane0 < DK);
    fence_proxy_async();
    fence_before_sync();
    named_bar(bar_id, 128);
    fence_after_sync();
    if (t == 0) {
      bulk_s2g(dst, sX2, 128 * 128);
      bulk_commit();
    }
  }
  if (t == 0) {
    if (ready) {
      // publish: the images are complete in global memory, then the flag
      bulk_wait_all();
      fence_proxy_async_global();
      store_release_gpu(ready + (size_t)slot * a.H + hq, 1);
    } else {
      // the bulk stores must have read shared memory before the unit's
      // buffers are reused; their global writes complete with the grid
      bulk_wait_read_all();
    }
  }

  // ---- tear-down ----
  fence_before_sync();
  named_bar(bar_id, 128);
  fence_after_sync();
  if (*abort_flag && tid == 0) atomicOr(a.flags, kFlagTimeout);
}


}  // namespace
}  // namespace gdn
