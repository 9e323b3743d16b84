// gdn_scan_tc.cu -- the serial-across-chunks scan kernel of the bf16 path, on
// the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// One CTA per (sequence, value head, NS-column slice of dv), 256 threads:
//  * warps 0-3 (the chain): thread t owns tensor-memory lane t and state row t
//    (key channel t).  The fp32 state slice S (dk x NS) lives in registers for
//    the whole sequence (register-resident state, stratat pull #1296, "What
//    this is"); an fp16 copy in shared memory is the B operand of the products
//    with S.  Per chunk (C rows, P1 and AqkT from the prep kernel's image):
//       D1 = [Kg; Qg] S                 one M=128 MMA (rows 0..63 keys,
//                                       64..127 queries), K = dk
//       Y  = diag(beta) (V - D1[keys])  -> fp16 B operand
//       D2 = P1 Y                       S <- diag(exp(b_last)) S + D2
//       D3 = AqkT Y                     O  = D1[queries] + D3 -> o
//    Two tensor-core round trips per chunk sit on the serial path; the O
//    products ride along.
//  * warps 4-7 (the producer) keep NST chunks in flight: one thread issues TMA
//    tile loads of the chunk's keys, queries (two 64-column panels each) and V
//    slice straight into the 128-byte-swizzled operand layout, plus a bulk copy
//    of the prep image; all threads fetch gates and beta with cp.async.  Once a
//    chunk has landed they convert keys and queries in place from bf16 to fp16
//    (gated per channel for KDA), form the per-row gate coefficients, and
//    publish the chunk to the chain.
// The split over dv slices manufactures the parallelism a (batch, head) grid
// lacks (ROCm/rocm-libraries PR #11223, "Notes for reviewers").  Operands are
// fp16 (11-bit mantissa) with fp32 accumulation; the state itself stays fp32.
// Every wait is bounded: a wait that runs out sets a status flag, after which
// all waits return at once and the kernel finishes with the same control flow
// in every thread (no hang, tensor memory freed).
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

constexpr int kThreads = 256;
constexpr int kChain = 128;  // chain threads (warps 0-3)
constexpr int NS = kScanTcSlice;
static_assert(NS == 64, "one 128-byte swizzle atom per V / S / Y row");

template <int C, int DK, int GATE, int NST>
struct ScanTcSmem {
  static constexpr int KQ = (DK / 64) * 128 * 128;  // [Kg; Qg], K-major, 128 rows
  static constexpr int PI = kPrepImageBytes;         // [P1; AqkT]
  static constexpr int VI = C * 128;                 // V slice, C rows of 64 bf16
  static constexpr int SI = (DK / 8) * 1024;         // S, MN-major, dk K-rows
  static constexpr int YI = 8 * 1024;                // Y, MN-major, 64 K-rows
  static constexpr int NRAW = GATE == 0 ? 2 * C : C * DK + C;  // gates, beta
  static constexpr int NCOEF = GATE == 0 ? 3 * C + 4 : C + DK;
  static constexpr int kKQ = 0;
  static constexpr int kP = kKQ + NST * KQ;
  static constexpr int kV = kP + NST * PI;
  static constexpr int kS = kV + NST * VI;
  static constexpr int kY = kS + SI;
  static constexpr int kRaw = kY + YI;
  static constexpr int kCoef = kRaw + NST * NRAW * 4;
  static constexpr int kBar = kCoef + NST * NCOEF * 4;
  static constexpr int kMisc = kBar + (3 * NST + 2) * 8;
  static constexpr int kBytes = kMisc + 16 + 1024;  // + alignment slack
  // bytes landing per chunk: [Kg; Qg] (GDN: the prep's fp16 image; KDA: two
  // TMA boxes per panel), the V slice and the prep image
  static constexpr uint32_t kTx = (GATE == 0 ? KQ : 2 * C * DK * 2) + C * NS * 2 + PI;
  static_assert(KQ % 1024 == 0 && PI % 1024 == 0 && VI % 1024 == 0 && SI % 1024 == 0,
                "1024-byte operand alignment");
  static_assert(kBytes <= 232448, "shared memory budget of one CTA");
};

template <int C, int DK, int GATE, int NST>
__global__ void __launch_bounds__(kThreads, 1)
gdn_scan_tc_kernel(const ScanArgs a, const __grid_constant__ ScanMaps maps) {
  using SM = ScanTcSmem<C, DK, GATE, NST>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM::kBar);
  // bars: full[NST] (data landed), ready[NST] (converted), empty[NST] (consumed),
  //       mma1, mma2
  const uint32_t bar_full = smem_addr(bars), bar_ready = smem_addr(bars + NST);
  const uint32_t bar_empty = smem_addr(bars + 2 * NST);
  const uint32_t bar_mma1 = smem_addr(bars + 3 * NST), bar_mma2 = smem_addr(bars + 3 * NST + 1);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + SM::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SM::kMisc + 4);

  const int n = blockIdx.x, hv = blockIdx.y, col0 = blockIdx.z * NS;
  const int hq = hv / (a.HV / a.H);
  const int tid = threadIdx.x, warp = tid >> 5;

  int start, end;
  bool ok = seq_ok(a.seq, n, start, end);
  if (a.seq.cu) ok = ok && __ldg(a.seq.cu) == 0 && __ldg(a.seq.cu + a.seq.n_seqs) == a.seq.Ttot;
  if (!ok) {  // uniform across the block: nothing allocated yet
    if (tid == 0) atomicOr(a.flags, kFlagBadSeqlens);
    return;
  }
  const int nchunks = (end - start + C - 1) / C;
  const int base = slot_base<C>(a.seq, n);

  // ---- set-up: barriers, tensor memory, zero rows no load ever writes ----
  if (tid == 0) {
    for (int s = 0; s < NST; s++) {
      mbar_init(bar_full + 8 * s, kChain + 1);
      mbar_init(bar_ready + 8 * s, kChain);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_mma1, 1);
    mbar_init(bar_mma2, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  constexpr uint32_t kTmemCols = 256;  // D1, D2, D3: 3 x NS columns
  if (warp == 0) tmem_alloc(smem_addr(tslot), kTmemCols);
  for (int i = tid; i < (NST * SM::KQ) / 16; i += kThreads)
    reinterpret_cast<uint4 *>(sm + SM::kKQ)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < SM::YI / 16; i += kThreads)
    reinterpret_cast<uint4 *>(sm + SM::kY)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tD1 = tmem, tD2 = tmem + NS, tD3 = tmem + 2 * NS;

  if (warp < 4) {
    // =====================================================================
    // chain
    // =====================================================================
    const int t = tid;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float s_reg[NS];
    const size_t hoff = ((size_t)n * a.HV + hv) * (size_t)DK * a.dv;
    if (t < DK) {
#pragma unroll
      for (int j = 0; j < NS; j += 4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.h0) v = __ldg(reinterpret_cast<const float4 *>(a.h0 + hoff + (size_t)t * a.dv + col0 + j));
        s_reg[j] = v.x; s_reg[j + 1] = v.y; s_reg[j + 2] = v.z; s_reg[j + 3] = v.w;
      }
    }
    auto write_state_image = [&]() {
      if (t < DK) {
#pragma unroll
        for (int ch = 0; ch < NS / 8; ch++) {
          uint4 pk;
          __half2 *h = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
          for (int i = 0; i < 4; i++) h[i] = __floats2half2_rn(s_reg[ch * 8 + 2 * i], s_reg[ch * 8 + 2 * i + 1]);
          *reinterpret_cast<uint4 *>(sm + SM::kS + mnmajor_chunk_off(t, ch, DK)) = pk;
        }
      }
    };
    write_state_image();
    fence_proxy_async();
    fence_before_sync();
    named_bar(1, kChain);

    constexpr uint32_t idesc = idesc_f16(128, NS, 0, 1);
    const uint32_t sS = smem_addr(sm + SM::kS), sY = smem_addr(sm + SM::kY);
    bool nonfinite = false;
    float o_part[NS];
    const bool key_warp = warp * 32 < C;
    const bool query_warp = warp >= 2 && (warp - 2) * 32 < C;

    // all NS columns of this thread's lane at column `col` (one wait)
    auto lane_row = [&](uint32_t col, float (&v)[NS]) {
      uint32_t r0[32], r1[32];
      tmem_ld32_nowait(col + lane_base, r0);
      tmem_ld32_nowait(col + lane_base + 32, r1);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; i++) { v[i] = __uint_as_float(r0[i]); v[32 + i] = __uint_as_float(r1[i]); }
    };
    // O of chunk cc = partial (Qg S) + AqkT Y, rounded to bf16 and stored
    auto output_rows = [&](int cc) {
      const int r = t - 64;
      const int t0 = start + cc * C;
      const int L = min(C, end - t0);
      float d[NS];
      lane_row(tD3, d);
      if (r < L) {
        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.o) + ((long)(t0 + r) * a.HV + hv) * a.dv + col0;
#pragma unroll
        for (int ch = 0; ch < NS / 8; ch++) {
          uint4 pk;
          __nv_bfloat162 *pb = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const float v0 = o_part[ch * 8 + 2 * i] + d[ch * 8 + 2 * i];
            const float v1 = o_part[ch * 8 + 2 * i + 1] + d[ch * 8 + 2 * i + 1];
            nonfinite |= !(isfinite(v0) && isfinite(v1));
            pb[i] = __floats2bfloat162_rn(v0, v1);
          }
          *reinterpret_cast<uint4 *>(orow + ch * 8) = pk;
        }
      }
    };

    for (int c = 0; c < nchunks; c++) {
      const int s = c % NST;
      const float *coef = reinterpret_cast<const float *>(sm + SM::kCoef + s * SM::NCOEF * 4);
      mbar_wait(bar_ready + 8 * s, (c / NST) & 1, abort_flag);

      // ---- D1 = [Kg; Qg] S ----
      if (t == 0) {
        fence_after_sync();
        const uint32_t sKQ = smem_addr(sm + SM::kKQ + s * SM::KQ);
#pragma unroll
        for (int k0 = 0; k0 < DK; k0 += 16) {
          const uint64_t ad = make_desc(sKQ + (k0 >> 6) * 16384 + (k0 & 63) * 2, 16, 1024);
          const uint64_t bd = make_desc(sS + (k0 >> 4) * 2048, (DK / 8) * 1024, 1024);
          mma_f16(tD1, ad, bd, idesc, k0 > 0 ? 1u : 0u);
        }
        mma_commit(bar_mma1);
      }
      // coefficients (read before the stage is handed back)
      float beta_r = 0.f, gam_r = 0.f, sgam_r = 0.f, dec = 0.f;
      if constexpr (GATE == 0) {
        const int r = t & 63;
        if (r < C) { beta_r = coef[r]; gam_r = coef[C + r]; sgam_r = coef[2 * C + r]; }
        dec = coef[3 * C];
      } else {
        if (t < C) beta_r = coef[t];
        if (t < DK) dec = coef[C + t];
      }
      // the previous chunk's output, while this chunk's first product runs
      if (query_warp && c > 0) output_rows(c - 1);
      mbar_wait(bar_mma1, c & 1, abort_flag);
      fence_after_sync();

      if (key_warp) {
        // key rows: Y = beta (V - gam X) -> fp16 image row t
        const unsigned char *vrow = sm + SM::kV + s * SM::VI + t * 128;
        float x[NS];
        lane_row(tD1, x);
#pragma unroll
        for (int ch = 0; ch < NS / 8; ch++) {
          const uint4 vv = *reinterpret_cast<const uint4 *>(vrow + ((ch ^ (t & 7)) << 4));
          const __nv_bfloat162 *vb = reinterpret_cast<const __nv_bfloat162 *>(&vv);
          uint4 pk;
          __half2 *ph = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const float2 vf = __bfloat1622float2(vb[i]);
            const float xa = GATE == 0 ? gam_r * x[ch * 8 + 2 * i] : x[ch * 8 + 2 * i];
            const float xb = GATE == 0 ? gam_r * x[ch * 8 + 2 * i + 1] : x[ch * 8 + 2 * i + 1];
            ph[i] = __floats2half2_rn(beta_r * (vf.x - xa), beta_r * (vf.y - xb));
          }
          *reinterpret_cast<uint4 *>(sm + SM::kY + mnmajor_chunk_off(t, ch, 64)) = pk;
        }
      } else if (query_warp) {
        // query rows: partial output of this chunk
        lane_row(tD1, o_part);
        if constexpr (GATE == 0) {
#pragma unroll
          for (int i = 0; i < NS; i++) o_part[i] *= sgam_r;
        }
      }
      fence_proxy_async();
      fence_before_sync();
      named_bar(1, kChain);

      // ---- D2 = P1 Y, D3 = AqkT Y ----
      if (t == 0) {
        fence_after_sync();
        const uint32_t sP = smem_addr(sm + SM::kP + s * SM::PI);
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16) {
          const uint64_t bd = make_desc(sY + (k0 >> 4) * 2048, 8 * 1024, 1024);
          mma_f16(tD2, make_desc(sP + k0 * 2, 16, 1024), bd, idesc, k0 > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16) {
          const uint64_t bd = make_desc(sY + (k0 >> 4) * 2048, 8 * 1024, 1024);
          mma_f16(tD3, make_desc(sP + 64 * 128 + k0 * 2, 16, 1024), bd, idesc, k0 > 0 ? 1u : 0u);
        }
        mma_commit(bar_mma2);
      }
      mbar_wait(bar_mma2, c & 1, abort_flag);
      fence_after_sync();
      if (t == 0) mbar_arrive(bar_empty + 8 * s);  // MMAs and reads of stage s are done

      if (t < DK) {
        float d[NS];
        lane_row(tD2, d);
#pragma unroll
        for (int i = 0; i < NS; i++) s_reg[i] = fmaf(dec, s_reg[i], d[i]);
        write_state_image();
      }
      fence_proxy_async();
      fence_before_sync();
      named_bar(1, kChain);
    }
    if (query_warp && nchunks > 0) output_rows(nchunks - 1);

    // ---- final state ----
    if (a.hT && t < DK) {
#pragma unroll
      for (int j = 0; j < NS; j += 4) {
        nonfinite |= !(isfinite(s_reg[j]) && isfinite(s_reg[j + 1]) && isfinite(s_reg[j + 2]) &&
                       isfinite(s_reg[j + 3]));
        *reinterpret_cast<float4 *>(a.hT + hoff + (size_t)t * a.dv + col0 + j) =
            make_float4(s_reg[j], s_reg[j + 1], s_reg[j + 2], s_reg[j + 3]);
      }
    }
    if (nonfinite) atomicOr(a.flags, kFlagNonfinite);
  } else {
    // =====================================================================
    // producer
    // =====================================================================
    const int pt = tid - kChain;
    // issue the loads of chunk c into stage c % NST
    auto issue = [&](int c) {
      const int s = c % NST;
      if (c >= NST) mbar_wait(bar_empty + 8 * s, ((c / NST) - 1) & 1, abort_flag);
      const int t0 = start + c * C;
      const int L = min(C, end - t0);
      const uint32_t full = bar_full + 8 * s;
      if (pt == 0) {
        mbar_arrive_expect_tx(full, SM::kTx);
        const uint32_t kq = smem_addr(sm + SM::kKQ + s * SM::KQ);
        if constexpr (GATE == 0) {
          // fp16 [K; Q] image written by the prep kernel
          bulk_g2s(kq, a.kq_images + ((size_t)(base + c) * a.H + hq) * SM::KQ, SM::KQ, full);
        } else {
#pragma unroll
          for (int p = 0; p < DK / 64; p++) {
            tma_load_3d(kq + p * 16384, &maps.k, p * 64, hq, t0, full);
            tma_load_3d(kq + p * 16384 + 64 * 128, &maps.q, p * 64, hq, t0, full);
          }
        }
        tma_load_3d(smem_addr(sm + SM::kV + s * SM::VI), &maps.v, col0, hv, t0, full);
        const unsigned char *src = reinterpret_cast<const unsigned char *>(a.tiles) +
                                   ((size_t)(base + c) * a.HV + hv) * kPrepImageBytes;
        bulk_g2s(smem_addr(sm + SM::kP + s * SM::PI), src, kPrepImageBytes, full);
      }
      float *raw = reinterpret_cast<float *>(sm + SM::kRaw + s * SM::NRAW * 4);
      if constexpr (GATE == 0) {
        if (pt < C) {
          const bool in = pt < L;
          const long row = in ? (long)(t0 + pt) : (long)t0;
          cp_async4(smem_addr(raw + pt), a.g + row * a.HV + hv, in ? 4u : 0u);
          cp_async4(smem_addr(raw + C + pt), a.beta + row * a.HV + hv, in ? 4u : 0u);
        }
      } else {
        for (int idx = pt; idx < C * DK / 4; idx += kChain) {
          const int r = idx / (DK / 4), c4 = (idx % (DK / 4)) * 4;
          const bool in = r < L;
          const long row = in ? (long)(t0 + r) : (long)t0;
          cp_async16(smem_addr(raw + r * DK + c4), a.g + (row * a.HV + hv) * DK + c4, in ? 16u : 0u);
        }
        if (pt < C) {
          const bool in = pt < L;
          const long row = in ? (long)(t0 + pt) : (long)t0;
          cp_async4(smem_addr(raw + C * DK + pt), a.beta + row * a.HV + hv, in ? 4u : 0u);
        }
      }
      cp_async_arrive_noinc(full);
    };

    // convert chunk c (landed) in place and publish it
    auto finish = [&](int c) {
      const int s = c % NST;
      const int t0 = start + c * C;
      const int L = min(C, end - t0);
      mbar_wait(bar_full + 8 * s, (c / NST) & 1, abort_flag);
      unsigned char *kq = sm + SM::kKQ + s * SM::KQ;
      float *raw = reinterpret_cast<float *>(sm + SM::kRaw + s * SM::NRAW * 4);
      float *coef = reinterpret_cast<float *>(sm + SM::kCoef + s * SM::NCOEF * 4);
      if constexpr (GATE == 0) {
        // keys and queries arrived as fp16 already; only the gate coefficients
        if (pt < 32) {
          const int lane = pt;
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
            coef[lane] = raw[C + lane];
            coef[C + lane] = gm;
            coef[2 * C + lane] = a.scale * gm;
          }
          if (lane + 32 < C) {
            const float gm = __expf(x1);
            coef[lane + 32] = raw[C + lane + 32];
            coef[C + lane + 32] = gm;
            coef[2 * C + lane + 32] = a.scale * gm;
          }
          if (lane == 0) coef[3 * C] = __expf(blast);
        }
      } else {
        // per key channel: cumulative gate -> exp in place; decay of the chunk
        if (pt < DK) {
          float run = 0.f;
          bool positive = false;
          for (int r = 0; r < C; r++) {
            const float gk = raw[r * DK + pt];
            positive |= gk > 0.f;
            run += gk;
            raw[r * DK + pt] = __expf(run);
          }
          coef[C + pt] = __expf(run);
          if (positive) atomicOr(a.flags, kFlagPositiveGate);
        }
        if (pt < C) coef[pt] = raw[C * DK + pt];
        named_bar(2, kChain);
        // gated keys / queries: bf16 -> fp16 (k exp(b), scale q exp(b)) in place
        constexpr int CH = (DK / 64) * 2 * C * 8;
        for (int idx = pt; idx < CH; idx += kChain) {
          const int p = idx / (2 * C * 8), rem = idx % (2 * C * 8);
          const int half = rem / (C * 8), r = (rem / 8) % C, chunk = rem % 8;
          const int row = half * 64 + r;
          uint4 *ptr = reinterpret_cast<uint4 *>(kq + p * 16384 + row * 128 + chunk * 16);
          const int col = p * 64 + ((chunk ^ (row & 7)) << 3);  // first channel of the chunk
          uint4 v = *ptr, out = make_uint4(0, 0, 0, 0);
          if (r < L) {
            const float mul = half ? a.scale : 1.f;
            const float *gm = raw + r * DK + col;
            const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&v);
            __half2 *h = reinterpret_cast<__half2 *>(&out);
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const float2 f = __bfloat1622float2(b[i]);
              h[i] = __floats2half2_rn(mul * f.x * gm[2 * i], mul * f.y * gm[2 * i + 1]);
            }
          }
          *ptr = out;
        }
      }
      fence_proxy_async();
      mbar_arrive(bar_ready + 8 * s);
    };

    for (int c = 0; c < NST - 1 && c < nchunks; c++) issue(c);
    for (int c = 0; c < nchunks; c++) {
      finish(c);
      if (c + NST - 1 < nchunks) issue(c + NST - 1);
    }
  }

  // ---- tear-down ----
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (*abort_flag && tid == 0) atomicOr(a.flags, kFlagTimeout);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int C, int DK, int GATE, int NST>
cudaError_t launch_one(const ScanArgs &a, const ScanMaps &maps, cudaStream_t stream) {
  using SM = ScanTcSmem<C, DK, GATE, NST>;
  auto kern = gdn_scan_tc_kernel<C, DK, GATE, NST>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (err != cudaSuccess) return err;
  kern<<<dim3(a.seq.n_seqs, a.HV, a.dv / NS), kThreads, SM::kBytes, stream>>>(a, maps);
  return cudaGetLastError();
}

template <int C, int DK>
cudaError_t dispatch_gate(const ScanArgs &a, const ScanMaps &m, int gate, cudaStream_t s) {
  // three stages in flight where shared memory allows (GDN), two for KDA,
  // whose per-channel gates take a stage's worth of room
  return gate ? launch_one<C, DK, 1, 2>(a, m, s) : launch_one<C, DK, 0, 3>(a, m, s);
}

}  // namespace

cudaError_t launch_scan_tc(const ScanArgs &a, const ScanMaps &maps, int chunk, int dk, int gate,
                           cudaStream_t stream) {
  if (chunk == 64 && dk == 128) return dispatch_gate<64, 128>(a, maps, gate, stream);
  if (chunk == 64 && dk == 64) return dispatch_gate<64, 64>(a, maps, gate, stream);
  if (chunk == 32 && dk == 128) return dispatch_gate<32, 128>(a, maps, gate, stream);
  if (chunk == 32 && dk == 64) return dispatch_gate<32, 64>(a, maps, gate, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
