// gdn_scan_la.cuh -- the serial-across-chunks scan of the bf16 scalar-gate
// (GDN) path as a device function over one block of its grid.  gdn_scan_la.cu
// launches it as its own kernel after the prep kernel; the lockstep kernel
// (gdn_lockstep.cu) runs it beside persistent prep warpgroups, loading each
// prep image once its ready flag is set.
//
// The chunk form (stratat pull #1296, "What this is": the state walk over
// chunks with W and U folded into per-chunk operands) needs, for chunk c with
// entering state S_c,
//   X_c = K_c S_c                      Y_c = diag(beta)(V_c - diag(gam) X_c)
//   S_{c+1} = d_c S_c + P1_c Y_c       O_c = scale diag(gam) Q_c S_c + AqkT_c Y_c
// (gam = exp(b), d_c = exp(b_last), P1 = K^T diag(exp(b_last - b)) T, all per
// chunk).  Computing X_c from S_c puts two tensor-core round trips on the
// serial path.  Expanding S_c instead gives
//   X_c = d_{c-1} (K_c S_{c-1}) + E_c Y_{c-1},   E_c = K_c P1_{c-1},
// with E_c state-independent (written by the prep kernel).  Per chunk c, in
// this order on the tensor pipe:
//   MMA1(c) = [E_c; AqkT_{c-1}] Y_{c-1}      -> D1[c%3]     (X_c part, O_{c-1} part)
//   MMA3(c) = [K_c; Q_{c-1}] S_{c-1}         -> D3[(c-1)&1] (X_c part, O_{c-1} part)
//   MMA2(c) = P1_{c-1} Y_{c-1}               -> D2          (state update)
// all M = 128, N = 64 (a dv slice), fp16 operands, fp32 accumulation in
// tensor memory.  The chain forms Y_c as soon as MMA1(c) and MMA3(c) are
// done, and only then S_c = d_{c-1} S_{c-1} + D2, whose fp16 image feeds
// MMA3(c + 1): the state update stays off the path from Y_{c-1} to Y_c,
// where MMA3(c) overlaps the chain's loads of chunk c's coefficients and V.
//
// One CTA per (sequence, value head, 64-column slice of dv), 384 threads,
// longest packed sequences first:
//  * warps 0-7 (the chain): warp w owns tensor-memory lanes 32 (w % 4) .. +31
//    and columns 32 (w / 4) .. +31 of the slice.  The fp32 state slice
//    (dk x 64) lives in registers for the whole sequence; an fp16 copy in
//    shared memory is the B operand of MMA3.  Lanes below C form Y (key rows),
//    lanes 64..64+C-1 form O (query rows), lanes below dk update the state.
//  * warp 8, one thread: issues every tensor-core product, the TMA loads of V
//    (a three-deep ring) and the bulk copies of the prep images (three deep).
//    Y is double-buffered (MMA2(c) may still read Y_{c-1} while Y_c is
//    written) and D1 triple-buffered (the query lanes read it one chunk late).
//  * warp 9: gates and beta by cp.async, cumulative gates and the per-row
//    coefficients (a four-deep ring); in the lockstep kernel also the prep
//    units' ready flags, acquired ahead and published in shared memory.
//  * warps 10-11: the [K_{c+1}; Q_c] operand (a two-deep ring): bulk copies of
//    the prep kernel's fp16 image; the first chunk's [K_0; Q_0] by TMA of the
//    bf16 tiles, converted in place.
// Every wait is bounded: a wait that runs out sets a status flag, after which
// all waits return at once and the kernel finishes with the same control flow
// in every thread (no hang, tensor memory freed).
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

constexpr int kChain = 256;       // warps 0-7
constexpr int kIssuerWarp = 8;
constexpr int kCoefWarp = 9;
constexpr int kKqWarp0 = 10;      // warps 10-11
constexpr int kKqThreads = 64;
constexpr int kThreads = 384;
constexpr int NS = kScanTcSlice;
constexpr int NH = NS / 2;  // columns per chain thread
static_assert(NS == 64, "one 128-byte swizzle atom per S / Y row");

template <int C, int DK>
struct LaSmem {
  static constexpr int NKQ = 2, NP = 3, NCF = 4, NV = 3;
  static constexpr int KQ = (DK / 64) * 16384;  // [K_{c+1}; Q_c], K-major, 128 rows
  static constexpr int PI = kLaImageBytes;       // [P1; E; AqkT]
  static constexpr int SI = (DK / 8) * 1024;     // S, MN-major, dk K-rows
  static constexpr int YI = 8 * 1024;            // Y, MN-major, 64 K-rows (x2, by chunk parity)
  static constexpr int VI = C * 128;             // V slice, C rows x 64 bf16 (x NV)
  // per chunk: raw gates and beta (2C), then beta, gam, scale*gam (3C), decay
  static constexpr int CF = (5 * C + 4) * 4;
  static constexpr int kKQ = 0;
  static constexpr int kP = kKQ + NKQ * KQ;
  static constexpr int kS = kP + NP * PI;
  static constexpr int kY = kS + SI;
  static constexpr int kV = kY + 2 * YI;
  static constexpr int kCf = kV + NV * VI;
  static constexpr int kBar = kCf + NCF * CF;
  enum {
    B_KQFULL = 0,
    B_KQREADY = B_KQFULL + NKQ,
    B_KQEMPTY = B_KQREADY + NKQ,
    B_PFULL = B_KQEMPTY + NKQ,
    B_CFFULL = B_PFULL + NP,
    B_CFREADY = B_CFFULL + NCF,
    B_CFEMPTY = B_CFREADY + NCF,
    B_MMA1 = B_CFEMPTY + NCF,  // three, by chunk index mod 3
    B_MMA2 = B_MMA1 + 3,
    B_MMA3 = B_MMA2 + 1,       // two, by chunk parity
    B_SREADY = B_MMA3 + 2,
    B_YREADY = B_SREADY + 1,
    B_VFULL = B_YREADY + 1,    // NV V buffers
    NBAR = B_VFULL + NV
  };
  static constexpr int kMisc = kBar + NBAR * 8;
  static constexpr int kUnits = kMisc + 12;  // lockstep: prep units published ready
  static constexpr int kUsed = kMisc + 16;
  // request 1 KB of alignment slack when it fits; otherwise the kernel checks
  // that the dynamic shared memory it received is already 1 KB aligned
  static constexpr int kSlack = kUsed + 1024 <= 232448 ? 1024 : 0;
  static constexpr int kBytes = kUsed + kSlack;
  static_assert(KQ % 1024 == 0 && PI % 1024 == 0 && SI % 1024 == 0 && VI % 1024 == 0,
                "1024-byte operand alignment");
  static_assert(kBar % 8 == 0, "mbarrier alignment");
  static_assert(kBytes <= 232448, "shared memory budget of one CTA");
};

// "Units 0 .. n - 1 are ready" in a shared-memory word, written by the
// coefficient warp after its gpu-scope acquire of each unit's flag (release /
// acquire at CTA scope), so that the threads that issue the bulk copies wait
// on shared memory instead of an L2 round trip each.
__device__ __forceinline__ void publish_units(uint32_t word, int n) {
  asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"(word), "r"(n) : "memory");
}
__device__ __forceinline__ int units_ready(uint32_t word) {
  int n;
  asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(n) : "r"(word) : "memory");
  return n;
}
// Bounded wait until unit j is published; false once the clock budget runs
// out or another wait of the block gave up.
__device__ __forceinline__ bool wait_unit(uint32_t word, int j, volatile int *abort) {
  if (units_ready(word) > j) return true;
  const long long t0 = clock64();
  while (true) {
    if (*abort) return false;
    if (units_ready(word) > j) return true;
    if (clock64() - t0 > 4000000000LL) {
      *abort = 1;
      return false;
    }
  }
}

// The scan of one block (sequence, value head, dv slice) of the grid, run by
// 384 threads on the LaSmem layout at `sm` (1 KB aligned).  With LOCK (the
// lockstep kernel, `ready` its flags), every prep image is loaded only once
// its (chunk slot, q/k head) flag is set: the coefficient warp acquires the
// flags and publishes them in shared memory for the threads that issue the
// copies.  Without LOCK (the split kernel) none of that code exists; the
// arithmetic is the same either way.
template <int C, int DK, bool LOCK = false>
__device__ __forceinline__ void scan_la_block(const ScanArgs &a, const ScanMaps &maps,
                                              int block, unsigned char *sm, const int *ready) {
  using SM = LaSmem<C, DK>;
  constexpr int NKQ = SM::NKQ, NP = SM::NP, NCF = SM::NCF;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = smem_addr(sm + SM::kBar);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + SM::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SM::kMisc + 4);

  // longest packed sequences first (scan_sequence)
  const int n_slices = a.dv / NS;
  const int rank = block / (a.HV * n_slices);
  const int hv = (block / n_slices) % a.HV, col0 = (block % n_slices) * NS;
  const int hq = hv / (a.HV / a.H);
  const int n = scan_sequence(a.seq, rank, reinterpret_cast<int *>(sm + SM::kMisc + 8));

  int start, end;
  bool ok = seq_ok(a.seq, n, start, end);
  if (a.seq.cu) ok = ok && __ldg(a.seq.cu) == 0 && __ldg(a.seq.cu + a.seq.n_seqs) == a.seq.Ttot;
  if (!ok) {  // uniform across the block: nothing allocated yet
    if (tid == 0) atomicOr(a.flags, kFlagBadSeqlens);
    return;
  }
  const int nch = (end - start + C - 1) / C;
  const int base = slot_base<C>(a.seq, n);
  constexpr int kKeyWarps = 2 * (C / 32);  // chain warps holding key rows

  // ---- set-up: barriers, tensor memory ----
  if (tid == 0) {
    for (int s = 0; s < NKQ; s++) {
      mbar_init(bar(SM::B_KQFULL + s), 1);
      mbar_init(bar(SM::B_KQREADY + s), kKqThreads);
      mbar_init(bar(SM::B_KQEMPTY + s), 1);
    }
    for (int s = 0; s < NP; s++) mbar_init(bar(SM::B_PFULL + s), 1);
    for (int s = 0; s < NCF; s++) {
      mbar_init(bar(SM::B_CFFULL + s), 32);
      mbar_init(bar(SM::B_CFREADY + s), 32);
      mbar_init(bar(SM::B_CFEMPTY + s), kChain / 32);
    }
    for (int i = 0; i < 3; i++) mbar_init(bar(SM::B_MMA1 + i), 1);
    for (int i = 0; i < 2; i++) mbar_init(bar(SM::B_MMA3 + i), 1);
    for (int i = 0; i < SM::NV; i++) mbar_init(bar(SM::B_VFULL + i), 1);
    mbar_init(bar(SM::B_MMA2), 1);
    mbar_init(bar(SM::B_SREADY), kChain / 32);
    mbar_init(bar(SM::B_YREADY), kKeyWarps);
    *abort_flag = 0;
    if constexpr (LOCK) publish_units(smem_addr(sm + SM::kUnits), 0);
    mbar_fence_init();
  }
  constexpr uint32_t kTmemCols = 512;  // D1 x3, D2, D3 x2: 6 x NS columns
  if (warp == 0) tmem_alloc(smem_addr(tslot), kTmemCols);
  for (int i = tid; i < 2 * SM::YI / 16; i += kThreads)
    reinterpret_cast<uint4 *>(sm + SM::kY)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tD1 = tmem, tD2 = tmem + 3 * NS, tD3 = tmem + 4 * NS;
  constexpr uint32_t idesc = idesc_f16(128, NS, 0, 1);

  if (warp < 8) {
    // =====================================================================
    // chain
    // =====================================================================
    const int q = warp & 3, hh = warp >> 2;
    const int t = q * 32 + lane;        // tensor-memory lane = state row / chunk row
    const int c0 = hh * NH;             // first column of this thread
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const bool key_warp = q * 32 < C;                       // lanes of key rows
    const bool query_warp = q >= 2 && (q - 2) * 32 < C;     // lanes of query rows
    const bool state_warp = q * 32 < DK;
    float s_reg[NH];
    const size_t hoff = ((size_t)n * a.HV + hv) * (size_t)DK * a.dv;
    if (state_warp) {
#pragma unroll
      for (int j = 0; j < NH; j += 4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.h0) v = __ldg(reinterpret_cast<const float4 *>(a.h0 + hoff + (size_t)t * a.dv + col0 + c0 + j));
        s_reg[j] = v.x; s_reg[j + 1] = v.y; s_reg[j + 2] = v.z; s_reg[j + 3] = v.w;
      }
    }
    auto write_state_image = [&]() {
#pragma unroll
      for (int ch = 0; ch < NH / 8; ch++) {
        uint4 pk;
        __half2 *h = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
        for (int i = 0; i < 4; i++) h[i] = __floats2half2_rn(s_reg[ch * 8 + 2 * i], s_reg[ch * 8 + 2 * i + 1]);
        *reinterpret_cast<uint4 *>(sm + SM::kS + mnmajor_chunk_off(t, c0 / 8 + ch, DK)) = pk;
      }
    };
    // the 32 columns of this thread's lane at tensor-memory column `col`
    auto lane_half = [&](uint32_t col, float (&v)[NH]) {
      uint32_t r[32];
      tmem_ld32_nowait(col + lane_base + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
    };
    // publish this warp's shared-memory / tensor-memory work to the issuer
    auto signal = [&](int b) {
      fence_proxy_async();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(b));
    };
    bool nonfinite = false;
    // ---- O_cc = scale gam Q_cc S_cc + AqkT_cc Y_cc (query lanes) ----
    // Q_cc S_cc is in D3[cc & 1] (MMA3(cc + 1)), AqkT_cc Y_cc in
    // D1[(cc + 1) % 3] (MMA1(cc + 1)).  The products that overwrite them,
    // MMA3(cc + 3) and MMA1(cc + 4), are issued only after SREADY(cc + 2),
    // which this thread joins after writing the output.  The
    // output of chunk cc is written at the top of iteration cc + 2, while
    // the tensor pipe runs the state products, so that its tensor-memory
    // reads and global stores stay out of the window in which the key lanes
    // form Y through shared memory.
    auto output = [&](int cc, float sg) {
      const int r = t - 64;
      const int t0 = start + cc * C;
      const int L = min(C, end - t0);
      float qs[NH], d[NH];
      lane_half(tD3 + (cc & 1) * NS, qs);
      lane_half(tD1 + ((cc + 1) % 3) * NS, d);
      if (r < L) {
        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.o) + ((long)(t0 + r) * a.HV + hv) * a.dv + col0 + c0;
#pragma unroll
        for (int ch = 0; ch < NH / 8; ch++) {
          uint4 pk;
          __nv_bfloat162 *pb = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const int j = ch * 8 + 2 * i;
            const float v0 = fmaf(sg, qs[j], d[j]);
            const float v1 = fmaf(sg, qs[j + 1], d[j + 1]);
            nonfinite |= !(isfinite(v0) && isfinite(v1));
            pb[i] = __floats2bfloat162_rn(v0, v1);
          }
          *reinterpret_cast<uint4 *>(orow + ch * 8) = pk;
        }
      }
    };

    if (nch > 0) {
      if (state_warp) write_state_image();
      signal(SM::B_SREADY);  // S_0
      float dec_prev = 1.f, sgam_prev = 0.f, sgam_prev2 = 0.f;
      for (int c = 0; c <= nch; c++) {
        // coefficients of chunk c (into registers, then the slot is handed back)
        float beta_r = 0.f, gam_r = 0.f, sgam_r = 0.f, dec_c = 0.f;
        if (c < nch) {
          const int s = c % NCF;
          mbar_wait(bar(SM::B_CFREADY + s), (c / NCF) & 1, abort_flag);
          const float *cf = reinterpret_cast<const float *>(sm + SM::kCf + s * SM::CF) + 2 * C;
          const int r = t & 63;
          if (r < C) { beta_r = cf[r]; gam_r = cf[C + r]; sgam_r = cf[2 * C + r]; }
          dec_c = cf[3 * C];
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(SM::B_CFEMPTY + s));
        }
        // this row of V_c into registers now, while the products of the
        // previous chunk run: shared memory is quiet here, and busy with the
        // state product's operand reads while Y_c is formed
        uint4 vv[NH / 8];
        if (key_warp && c < nch) {
          mbar_wait(bar(SM::B_VFULL + c % SM::NV), (c / SM::NV) & 1, abort_flag);
          const unsigned char *vrow = sm + SM::kV + (c % SM::NV) * SM::VI + t * 128;
#pragma unroll
          for (int ch = 0; ch < NH / 8; ch++)
            vv[ch] = *reinterpret_cast<const uint4 *>(vrow + (((c0 / 8 + ch) ^ (t & 7)) << 4));
        }
        if (query_warp && c >= 2) output(c - 2, sgam_prev2);
        // X_c's products: E_c Y_{c-1} (MMA1(c)) and K_c S_{c-1} (MMA3(c); chunk
        // 0: K_0 S_0)
        if (c >= 1) mbar_wait(bar(SM::B_MMA1 + c % 3), ((c - 1) / 3) & 1, abort_flag);
        mbar_wait(bar(SM::B_MMA3 + ((c - 1) & 1)), (c >> 1) & 1, abort_flag);
        fence_after_sync();
        const uint32_t d3 = tD3 + ((c - 1) & 1) * NS, d1 = tD1 + (c % 3) * NS;

        if (key_warp && c < nch) {
          // ---- Y_c = beta (V - gam X), X = d_{c-1} K_c S_{c-1} + E_c Y_{c-1} ----
          float x[NH];
          lane_half(d3, x);
          if (c >= 1) {
            float e[NH];
            lane_half(d1, e);
#pragma unroll
            for (int i = 0; i < NH; i++) x[i] = fmaf(dec_prev, x[i], e[i]);
          }
          unsigned char *ybuf = sm + SM::kY + (c & 1) * SM::YI;
#pragma unroll
          for (int ch = 0; ch < NH / 8; ch++) {
            const __nv_bfloat162 *vb = reinterpret_cast<const __nv_bfloat162 *>(&vv[ch]);
            uint4 pk;
            __half2 *ph = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const float2 vf = __bfloat1622float2(vb[i]);
              ph[i] = __floats2half2_rn(beta_r * (vf.x - gam_r * x[ch * 8 + 2 * i]),
                                        beta_r * (vf.y - gam_r * x[ch * 8 + 2 * i + 1]));
            }
            *reinterpret_cast<uint4 *>(ybuf + mnmajor_chunk_off(t, c0 / 8 + ch, 64)) = pk;
          }
          signal(SM::B_YREADY);
        }
        // ---- state, after Y_c: S_c = d_{c-1} S_{c-1} + P1_{c-1} Y_{c-1} ----
        // (its product MMA3(c + 1) is needed only by X_{c+1})
        if (c >= 1) {
          mbar_wait(bar(SM::B_MMA2), (c - 1) & 1, abort_flag);
          fence_after_sync();
          if (state_warp) {
            float d[NH];
            lane_half(tD2, d);
#pragma unroll
            for (int i = 0; i < NH; i++) s_reg[i] = fmaf(dec_prev, s_reg[i], d[i]);
            if (c < nch) write_state_image();
          }
          if (c < nch) signal(SM::B_SREADY);
        }
        dec_prev = dec_c;
        sgam_prev2 = sgam_prev;
        sgam_prev = sgam_r;
      }
      if (query_warp) output(nch - 1, sgam_prev2);
    }

    // ---- final state ----
    if (a.hT && state_warp) {
#pragma unroll
      for (int j = 0; j < NH; j += 4) {
        nonfinite |= !(isfinite(s_reg[j]) && isfinite(s_reg[j + 1]) && isfinite(s_reg[j + 2]) &&
                       isfinite(s_reg[j + 3]));
        *reinterpret_cast<float4 *>(a.hT + hoff + (size_t)t * a.dv + col0 + c0 + j) =
            make_float4(s_reg[j], s_reg[j + 1], s_reg[j + 2], s_reg[j + 3]);
      }
    }
    if (nonfinite) atomicOr(a.flags, kFlagNonfinite);
  } else if (warp == kIssuerWarp) {
    // =====================================================================
    // issuer: tensor-core products, V and prep-image loads
    // =====================================================================
    if (lane == 0 && nch > 0) {
      const uint32_t sS = smem_addr(sm + SM::kS), sY = smem_addr(sm + SM::kY);
      auto issue_v = [&](int cc) {  // V slice of chunk cc -> buffer cc % NV
        const uint32_t b = bar(SM::B_VFULL + cc % SM::NV);
        mbar_arrive_expect_tx(b, SM::VI);
        tma_load_3d(smem_addr(sm + SM::kV + (cc % SM::NV) * SM::VI), &maps.v, col0, hv, start + cc * C, b);
      };
      auto issue_p = [&](int j) {  // prep image of chunk j -> slot j % NP
        if constexpr (LOCK) {
          wait_unit(smem_addr(sm + SM::kUnits), j, abort_flag);
          fence_proxy_async_global();
        }
        const uint32_t b = bar(SM::B_PFULL + j % NP);
        mbar_arrive_expect_tx(b, SM::PI);
        const unsigned char *src = reinterpret_cast<const unsigned char *>(a.tiles) +
                                   ((size_t)(base + j) * a.HV + hv) * SM::PI;
        bulk_g2s(smem_addr(sm + SM::kP + (j % NP) * SM::PI), src, SM::PI, b);
      };
      // MMA3 from KQ entry e (entry e holds [K_e; Q_{max(e-1,0)}]) into D3[buf]
      auto mma3 = [&](int e, int buf) {
        const int s = e % NKQ;
        mbar_wait(bar(SM::B_KQREADY + s), (e / NKQ) & 1, abort_flag);
        fence_after_sync();
        const uint32_t sKQ = smem_addr(sm + SM::kKQ + s * SM::KQ);
#pragma unroll
        for (int k0 = 0; k0 < DK; k0 += 16) {
          const uint64_t ad = make_desc(sKQ + (k0 >> 6) * 16384 + (k0 & 63) * 2, 16, 1024);
          const uint64_t bd = make_desc(sS + (k0 >> 4) * 2048, (DK / 8) * 1024, 1024);
          mma_f16(tD3 + buf * NS, ad, bd, idesc, k0 > 0 ? 1u : 0u);
        }
        mma_commit(bar(SM::B_MMA3 + buf));
        mma_commit(bar(SM::B_KQEMPTY + s));
      };

      for (int cc = 0; cc < SM::NV && cc < nch; cc++) issue_v(cc);
      issue_p(0);
      if (nch > 1) issue_p(1);
      mbar_wait(bar(SM::B_SREADY), 0, abort_flag);  // S_0 image
      mma3(0, 1);  // [K_0; Q_0] S_0 -> D3[1] (read as "chunk -1")
      // Per chunk, in this order: MMA1(c) and MMA3(c) give X_c (the serial
      // path), MMA2(c) the next state (needed only after Y_c).
      for (int c = 1; c <= nch; c++) {
        mbar_wait(bar(SM::B_YREADY), (c - 1) & 1, abort_flag);  // Y_{c-1}, V_{c-1} consumed
        const int ps = (c - 1) % NP;
        mbar_wait(bar(SM::B_PFULL + ps), ((c - 1) / NP) & 1, abort_flag);
        fence_after_sync();
        const uint32_t sP = smem_addr(sm + SM::kP + ps * SM::PI);
        const uint32_t sYp = sY + ((c - 1) & 1) * SM::YI;  // Y_{c-1}
#pragma unroll
        for (int k0 = 0; k0 < C; k0 += 16) {
          const uint64_t bd = make_desc(sYp + (k0 >> 4) * 2048, 8 * 1024, 1024);
          mma_f16(tD1 + (c % 3) * NS, make_desc(sP + 128 * 128 + k0 * 2, 16, 1024), bd, idesc,
                  k0 > 0 ? 1u : 0u);
        }
        mma_commit(bar(SM::B_MMA1 + c % 3));
        // S_{c-1} image (chunk 1: S_0, waited above)
        mbar_wait(bar(SM::B_SREADY), (c - 1) & 1, abort_flag);
        mma3(c, (c - 1) & 1);  // [K_c; Q_{c-1}] S_{c-1}
#pragma unroll
        for (int k0 = 0; k0 < C; k0 += 16) {
          const uint64_t bd = make_desc(sYp + (k0 >> 4) * 2048, 8 * 1024, 1024);
          mma_f16(tD2, make_desc(sP + k0 * 2, 16, 1024), bd, idesc, k0 > 0 ? 1u : 0u);
        }
        mma_commit(bar(SM::B_MMA2));
        // loads for later chunks, off the serial path: V of chunk c + 2 into
        // the buffer V_{c-1} left; the prep image of chunk c + 1 into the slot
        // of chunk c - 2, once MMA1(c) is done (the pipe runs in order, so
        // MMA2(c - 1), that slot's last reader, is done too)
        if (c + 2 < nch) issue_v(c + 2);
        if (c + 1 < nch) {
          mbar_wait(bar(SM::B_MMA1 + c % 3), ((c - 1) / 3) & 1, abort_flag);
          issue_p(c + 1);
        }
      }
    }
  } else if (warp == kCoefWarp) {
    // =====================================================================
    // coefficients: b = cumsum g; beta, gam = exp(b), scale gam, exp(b_last)
    // =====================================================================
    auto issue_cf = [&](int c) {
      const int s = c % NCF;
      if (c >= NCF) mbar_wait(bar(SM::B_CFEMPTY + s), ((c / NCF) - 1) & 1, abort_flag);
      const int t0 = start + c * C;
      const int L = min(C, end - t0);
      float *raw = reinterpret_cast<float *>(sm + SM::kCf + s * SM::CF);
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const int r = lane + 32 * h;
        if (r < C) {
          const bool in = r < L;
          const long row = in ? (long)(t0 + r) : (long)t0;
          cp_async4(smem_addr(raw + r), a.g + row * a.HV + hv, in ? 4u : 0u);
          cp_async4(smem_addr(raw + C + r), a.beta + row * a.HV + hv, in ? 4u : 0u);
        }
      }
      cp_async_arrive_noinc(bar(SM::B_CFFULL + s));
    };
    auto finish_cf = [&](int c) {
      const int s = c % NCF;
      mbar_wait(bar(SM::B_CFFULL + s), (c / NCF) & 1, abort_flag);
      const float *raw = reinterpret_cast<const float *>(sm + SM::kCf + s * SM::CF);
      float *cf = reinterpret_cast<float *>(sm + SM::kCf + s * SM::CF) + 2 * C;
      const float g0 = lane < C ? raw[lane] : 0.f;
      const float g1 = lane + 32 < C ? raw[lane + 32] : 0.f;
      if (__any_sync(0xffffffffu, g0 > 0.f || g1 > 0.f) && lane == 0) atomicOr(a.flags, kFlagPositiveGate);
      float x0 = g0, x1 = g1;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, x0, d);
        const float y1 = __shfl_up_sync(0xffffffffu, x1, d);
        if (lane >= d) { x0 += y0; x1 += y1; }
      }
      x1 += __shfl_sync(0xffffffffu, x0, 31);
      const float blast = __shfl_sync(0xffffffffu, C > 32 ? x1 : x0, (C - 1) & 31);
      if (lane < C) {
        const float gm = __expf(x0);
        cf[lane] = raw[C + lane];
        cf[C + lane] = gm;
        cf[2 * C + lane] = a.scale * gm;
      }
      if (lane + 32 < C) {
        const float gm = __expf(x1);
        cf[lane + 32] = raw[C + lane + 32];
        cf[C + lane + 32] = gm;
        cf[2 * C + lane + 32] = a.scale * gm;
      }
      if (lane == 0) cf[3 * C] = __expf(blast);
      mbar_arrive(bar(SM::B_CFREADY + s));
    };
    if constexpr (!LOCK) {
      for (int c = 0; c < NCF - 1 && c < nch; c++) issue_cf(c);
      for (int c = 0; c < nch; c++) {
        finish_cf(c);
        if (c + NCF - 1 < nch) issue_cf(c + NCF - 1);
      }
    } else {
      // lockstep: unit j (the prep images of chunk j) must be published
      // before its bulk copies, units 0..2 first and then j + 3 with the
      // coefficients of chunk j, about two chunks ahead.  When it is not yet,
      // the 32 lanes each acquire the flag of one of the next 32 units and the
      // ready prefix is published at once: one L2 round trip for up to 32
      // units.
      const uint32_t units_word = smem_addr(sm + SM::kUnits);
      int published = 0;
      auto relay = [&](int j) {
        if (j >= nch) return;
        const long long t0 = clock64();
        while (published <= j) {
          if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;  // uniform across the warp
          const int u = published + lane;
          const bool set = u >= nch || load_acquire_gpu(ready + (size_t)(base + u) * a.H + hq) != 0;
          const unsigned unset = __ballot_sync(0xffffffffu, !set);
          __syncwarp();  // the lanes' acquires before lane 0's release
          const int n = min(published + (unset ? __ffs(unset) - 1 : 32), nch);
          if (n > published) {
            published = n;
            if (lane == 0) publish_units(units_word, n);
          } else if (clock64() - t0 > 4000000000LL) {
            if (lane == 0) *abort_flag = 1;
            __syncwarp();
          } else {
            __nanosleep(100);
          }
        }
      };
      for (int j = 0; j < 3; j++) relay(j);
      for (int c = 0; c < NCF - 1 && c < nch; c++) issue_cf(c);
      for (int c = 0; c < nch; c++) {
        finish_cf(c);
        if (c + NCF - 1 < nch) issue_cf(c + NCF - 1);
        relay(c + 3);
      }
    }
  } else {
    // =====================================================================
    // keys and queries: entry e = [K_e; Q_{max(e-1,0)}] for e = 0..nch
    // (entry e feeds MMA3 of chunk e - 1).  Entry e >= 1 is the prep image
    // of chunk e - 1; entry 0 ([K_0; Q_0]) comes as bf16 tiles.
    // =====================================================================
    const int kt = tid - kKqWarp0 * 32;
    auto issue_kq = [&](int e) {
      const int s = e % NKQ;
      if (e >= NKQ) mbar_wait(bar(SM::B_KQEMPTY + s), ((e / NKQ) - 1) & 1, abort_flag);
      if (kt == 0) {
        const uint32_t b = bar(SM::B_KQFULL + s);
        const uint32_t kq = smem_addr(sm + SM::kKQ + s * SM::KQ);
        if (e > 0) {
          if constexpr (LOCK) {
            wait_unit(smem_addr(sm + SM::kUnits), e - 1, abort_flag);
            fence_proxy_async_global();
          }
          mbar_arrive_expect_tx(b, SM::KQ);
          bulk_g2s(kq, a.kq_images + ((size_t)(base + e - 1) * a.H + hq) * SM::KQ, SM::KQ, b);
        } else {
          mbar_arrive_expect_tx(b, 2 * (DK / 64) * C * 128);
#pragma unroll
          for (int p = 0; p < DK / 64; p++) {
            tma_load_3d(kq + p * 16384, &maps.k, p * 64, hq, start, b);
            tma_load_3d(kq + p * 16384 + 64 * 128, &maps.q, p * 64, hq, start, b);
          }
        }
      }
    };
    auto finish_kq = [&](int e) {
      const int s = e % NKQ;
      mbar_wait(bar(SM::B_KQFULL + s), (e / NKQ) & 1, abort_flag);
      if (e == 0) {
        // bf16 -> fp16 in place; rows beyond the tokens (and rows >= C) -> 0
        const int L0 = min(C, end - start);
        unsigned char *kq = sm + SM::kKQ + s * SM::KQ;
        constexpr int CH = (DK / 64) * 128 * 8;
        for (int idx = kt; idx < CH; idx += kKqThreads) {
          const int p = idx >> 10, row = (idx >> 3) & 127, chunk = idx & 7;
          uint4 *ptr = reinterpret_cast<uint4 *>(kq + p * 16384 + row * 128 + chunk * 16);
          uint4 out = make_uint4(0, 0, 0, 0);
          if ((row & 63) < L0) {
            const uint4 v = *ptr;
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
        fence_proxy_async();
      }
      mbar_arrive(bar(SM::B_KQREADY + s));
    };
    if (nch > 0) {
      for (int e = 0; e < NKQ && e <= nch; e++) issue_kq(e);
      for (int e = 0; e <= nch; e++) {
        finish_kq(e);
        if (e + NKQ <= nch) issue_kq(e + NKQ);
      }
    }
  }

  // ---- tear-down ----
  if (*abort_flag && tid == 0) {
    // a wait gave up: let copies and products still in flight land before the
    // shared and tensor memory are released (bounded, about 10 ms)
    const long long t0 = clock64();
    while (clock64() - t0 < 20000000LL) {
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (*abort_flag && tid == 0) atomicOr(a.flags, kFlagTimeout);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}


}  // namespace
}  // namespace gdn
