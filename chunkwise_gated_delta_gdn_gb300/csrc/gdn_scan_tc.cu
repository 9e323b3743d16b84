// gdn_scan_tc.cu -- the serial-across-chunks scan kernel of the bf16
// per-key-gate (KDA) path, on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory).  The scalar-gate path runs the lookahead
// scan of gdn_scan_la.cu.
//
// One CTA per (sequence, value head, NS-column slice of dv), 384 threads:
//  * warps 0-7 (the chain): warp w owns tensor-memory lanes / state rows
//    32 (w % 4) .. +31 (key channels) and columns 32 (w / 4) .. +31 of the
//    slice.  The fp32 state slice S (dk x NS) lives in registers for the whole
//    sequence (register-resident state, stratat pull #1296, "What this is");
//    an fp16 copy in shared memory is the B operand of the products with S.
//    Per chunk c (C rows, P1 and AqkT from the prep kernel's image):
//       D1[c&1] = [Kg; Qg] S          one M=128 MMA (key rows from 0, query
//                                     rows from C at chunk 32, from 64 at
//                                     chunk 64), K = dk
//       Y       = diag(beta)(V - D1[keys])       -> fp16 B operand Y[c&1]
//       D2      = P1 Y                S <- diag(exp(b_last)) S + D2
//       D3      = AqkT Y              issued right behind D2; it runs during
//                                     the state update, off the serial path
//       O       = D1[queries] + D3               -> o, during D1 of chunk c+1
//    (Kg = k e^b and Qg = scale q e^b per key channel, gated by the prep
//    kernel; the state decays per key channel, S <- diag(e^{b_last}) S.)
//    Two tensor-core round trips per chunk sit on the serial path.
//  * warps 8-11 (the producer) keep NST chunks in flight: one thread issues
//    bulk copies of the chunk's gated fp16 [Kg; Qg] image and of its [P1;
//    AqkT] image, both written by the prep kernel; cp.async brings beta and
//    the chunk's per-channel decay (also from the prep kernel).
// V arrives by TMA into a two-deep ring of its own, two chunks ahead of its
// use (issued by the chain as soon as a buffer has been consumed).  The split
// over dv slices manufactures the parallelism a (batch, head) grid lacks
// (ROCm/rocm-libraries PR #11223, "Notes for reviewers").
// Operands are fp16 (11-bit mantissa) with fp32 accumulation; the state itself
// stays fp32.  Every wait is bounded: a wait that runs out sets a status flag,
// after which all waits return at once and the kernel finishes with the same
// control flow in every thread (no hang, tensor memory freed).
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

constexpr int kChain = 256;  // chain threads (warps 0-7)
constexpr int kProd = 128;   // producer threads (warps 8-11)
constexpr int kThreads = kChain + kProd;
constexpr int NS = kScanTcSlice;
constexpr int NH = NS / 2;  // columns per chain thread
static_assert(NS == 64, "one 128-byte swizzle atom per S / Y row");

template <int C, int DK, int NST>
struct ScanTcSmem {
  static constexpr int KQ = (DK / 64) * 128 * 128;  // [Kg; Qg] stage, K-major, 128 rows per panel
  // The prep writes the image compactly at chunk 32 (per panel the C key rows,
  // then the C query rows: query lanes C..2C-1), at chunk 64 as 128 rows with
  // the queries from row 64; the stage keeps 128 rows per panel so that the
  // M = 128 product never reads past it.
  static constexpr bool COMPACT = C == 32;
  static constexpr int Q0 = COMPACT ? C : 64;          // first query row / lane
  static constexpr int KQP = COMPACT ? 2 * C * 128 : 128 * 128;  // bytes of one panel
  static constexpr int KQL = (DK / 64) * KQP;          // bytes copied per chunk
  static constexpr int PI = kPrepImageBytes;         // [P1; AqkT]
  static constexpr int SI = (DK / 8) * 1024;         // S, MN-major, dk K-rows
  static constexpr int YI = 8 * 1024;                // Y, MN-major, 64 K-rows (x2)
  static constexpr int NRAW = DK + C;   // decays, beta as landed
  static constexpr int NCOEF = C + DK;  // beta, decays
  static constexpr int kKQ = 0;
  static constexpr int kP = kKQ + NST * KQ;
  static constexpr int kS = kP + NST * PI;
  static constexpr int kY = kS + SI;
  static constexpr int VI = C * 128;                 // V slice, C rows x 64 bf16 (x2)
  static constexpr int kV = kY + 2 * YI;
  static constexpr int kRaw = kV + 2 * VI;
  static constexpr int kCoef = kRaw + NST * NRAW * 4;
  static constexpr int kBar = kCoef + NST * NCOEF * 4;
  static constexpr int kMisc = kBar + (3 * NST + 5) * 8;
  static constexpr int kUsed = kMisc + 16;
  // request 1 KB of alignment slack when it fits; otherwise the kernel checks
  // that the dynamic shared memory it received is already 1 KB aligned
  static constexpr int kSlack = kUsed + 1024 <= 232448 ? 1024 : 0;
  static constexpr int kBytes = kUsed + kSlack;
  // bytes landing per chunk: [Kg; Qg] (GDN: the prep's image; KDA: two TMA
  // boxes per panel) and the prep image
  // the [P1; AqkT] image: at chunk 32 its 10 KB form (32 columns per row, the
  // 64-byte swizzle), else 192 rows of 64 columns; the slot keeps 24 KB
  static constexpr int PL = COMPACT ? kPrepImage32Bytes : kPrepImageBytes;
  static constexpr uint32_t kTx = KQL + PL;
  static_assert(KQ % 1024 == 0 && PI % 1024 == 0 && SI % 1024 == 0 && VI % 1024 == 0,
                "1024-byte operand alignment");
  static_assert(kBytes <= 232448, "shared memory budget of one CTA");
};

template <int C, int DK, int NST>
__global__ void __launch_bounds__(kThreads, 1)
gdn_scan_tc_kernel(const ScanArgs a, const __grid_constant__ ScanMaps maps) {
  using SM = ScanTcSmem<C, DK, NST>;
  extern __shared__ unsigned char smem_raw[];
  // 1 KB-aligned base, as an offset into the shared array (the compiler then
  // knows every access below is to shared memory)
  unsigned char *sm = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (sm - smem_raw > SM::kSlack) {  // dynamic shared memory not aligned as needed
    if (tid == 0) atomicOr(a.flags, kFlagLaunchConfig);
    return;
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM::kBar);
  // bars: full[NST] (data landed), ready[NST] (published), empty[NST]
  //       (consumed), mma1, mma2, mma3, vfull[2]
  const uint32_t bar_full = smem_addr(bars), bar_ready = smem_addr(bars + NST);
  const uint32_t bar_empty = smem_addr(bars + 2 * NST);
  const uint32_t bar_mma1 = smem_addr(bars + 3 * NST), bar_mma2 = bar_mma1 + 8, bar_mma3 = bar_mma1 + 16;
  const uint32_t bar_v = bar_mma1 + 24;  // two V buffers
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + SM::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SM::kMisc + 4);

  // longest packed sequences first (scan_sequence)
  const int n_slices = a.dv / NS;
  const int hv = (blockIdx.x / n_slices) % a.HV, col0 = (blockIdx.x % n_slices) * NS;
  const int n = scan_sequence(a.seq, blockIdx.x / (a.HV * n_slices),
                              reinterpret_cast<int *>(sm + SM::kMisc + 8));

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
      mbar_init(bar_full + 8 * s, kProd + 1);
      mbar_init(bar_ready + 8 * s, kProd);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_mma1, 1);
    mbar_init(bar_mma2, 1);
    mbar_init(bar_mma3, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_v + 8, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  constexpr uint32_t kTmemCols = 256;  // D1 x2, D2, D3: 4 x NS columns
  if (warp == 0) tmem_alloc(smem_addr(tslot), kTmemCols);
  for (int i = tid; i < (2 * SM::YI) / 16; i += kThreads)
    reinterpret_cast<uint4 *>(sm + SM::kY)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tD1 = tmem, tD2 = tmem + 2 * NS, tD3 = tmem + 3 * NS;

  if (warp < 8) {
    // =====================================================================
    // chain
    // =====================================================================
    const int q = warp & 3, hh = warp >> 2;
    const int t = q * 32 + lane;        // tensor-memory lane = state row / chunk row
    const int c0 = hh * NH;             // first column of this thread
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const bool key_warp = q * 32 < C;                       // lanes of key rows
    const bool query_warp = q * 32 >= SM::Q0 && q * 32 - SM::Q0 < C;  // lanes of query rows
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
    if (state_warp) write_state_image();
    // V slice of chunk cc -> V buffer cc & 1 (TMA, issued by one thread)
    auto issue_v = [&](int cc) {
      const uint32_t bar = bar_v + 8 * (cc & 1);
      mbar_arrive_expect_tx(bar, SM::VI);
      tma_load_3d(smem_addr(sm + SM::kV + (cc & 1) * SM::VI), &maps.v, col0, hv, start + cc * C, bar);
    };
    if (tid == 0) {
      if (nchunks > 0) issue_v(0);
      if (nchunks > 1) issue_v(1);
    }
    fence_proxy_async();
    fence_before_sync();
    named_bar(1, kChain);

    constexpr uint32_t idesc = idesc_f16(128, NS, 0, 1);
    const uint32_t sS = smem_addr(sm + SM::kS), sY = smem_addr(sm + SM::kY);
    bool nonfinite = false;

    // the 32 columns of this thread's lane at tensor-memory column `col`
    auto lane_half = [&](uint32_t col, float (&v)[NH]) {
      uint32_t r[32];
      tmem_ld32_nowait(col + lane_base + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
    };
    // O of chunk cc = scale gam Qg S (D1[cc&1], query lanes) + AqkT Y (D3)
    auto output_rows = [&](int cc) {
      const int r = t - SM::Q0;
      const int t0 = start + cc * C;
      const int L = min(C, end - t0);
      float qs[NH], d[NH];
      lane_half(tD1 + (cc & 1) * NS, qs);
      lane_half(tD3, d);
      if (r < L) {
        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.o) + ((long)(t0 + r) * a.HV + hv) * a.dv + col0 + c0;
#pragma unroll
        for (int ch = 0; ch < NH / 8; ch++) {
          uint4 pk;
          __nv_bfloat162 *pb = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const int j = ch * 8 + 2 * i;
            const float v0 = qs[j] + d[j];
            const float v1 = qs[j + 1] + d[j + 1];
            nonfinite |= !(isfinite(v0) && isfinite(v1));
            pb[i] = __floats2bfloat162_rn(v0, v1);
          }
          *reinterpret_cast<uint4 *>(orow + ch * 8) = pk;
        }
      }
    };
    auto issue_o_intra = [&](int cc) {  // D3 = AqkT Y[cc&1]
      const uint32_t sP = smem_addr(sm + SM::kP + (cc % NST) * SM::PI);
#pragma unroll
      for (int k0 = 0; k0 < C; k0 += 16) {  // K = C: rows of Y beyond C are zero
        const uint64_t bd = make_desc(sY + (cc & 1) * SM::YI + (k0 >> 4) * 2048, 8 * 1024, 1024);
        // A from image row 128 - Q0: Aqk T row r lands in lane Q0 + r, the
        // query lane of row r (rows past the image read what follows it in
        // shared memory and land in lanes never read)
        const uint64_t ad = SM::COMPACT ? make_desc_sw64(sP + (128 - SM::Q0) * 64 + k0 * 2, 512)
                                        : make_desc(sP + (128 - SM::Q0) * 128 + k0 * 2, 16, 1024);
        mma_f16(tD3, ad, bd, idesc, k0 > 0 ? 1u : 0u);
      }
      mma_commit(bar_mma3);
    };

    for (int c = 0; c < nchunks; c++) {
      const int s = c % NST;
      const float *coef = reinterpret_cast<const float *>(sm + SM::kCoef + s * SM::NCOEF * 4);
      mbar_wait(bar_ready + 8 * s, (c / NST) & 1, abort_flag);

      // ---- D1[c&1] = [Kg; Qg] S; then the previous chunk's O-intra ----
      if (tid == 0) {
        fence_after_sync();
        const uint32_t sKQ = smem_addr(sm + SM::kKQ + s * SM::KQ);
#pragma unroll
        for (int k0 = 0; k0 < DK; k0 += 16) {
          const uint64_t ad = make_desc(sKQ + (k0 >> 6) * SM::KQP + (k0 & 63) * 2, 16, 1024);
          const uint64_t bd = make_desc(sS + (k0 >> 4) * 2048, (DK / 8) * 1024, 1024);
          mma_f16(tD1 + (c & 1) * NS, ad, bd, idesc, k0 > 0 ? 1u : 0u);
        }
        mma_commit(bar_mma1);
      }
      // coefficients of this chunk (read before the stage is handed back)
      float beta_r = 0.f, dec = 0.f;
      if (t < C) beta_r = coef[t];
      if (t < DK) dec = coef[C + t];
      // the previous chunk's output and its stage, while D1 runs
      if (c > 0) {
        mbar_wait(bar_mma3, (c - 1) & 1, abort_flag);
        fence_after_sync();
        // every product that read stage (c - 1) % NST has completed
        if (tid == 0) mbar_arrive(bar_empty + 8 * ((c - 1) % NST));
        if (query_warp) output_rows(c - 1);
      }
      mbar_wait(bar_mma1, c & 1, abort_flag);
      fence_after_sync();

      if (key_warp) {
        // key rows: Y = beta (V - gam X) -> fp16 image row t, this thread's columns
        float x[NH];
        lane_half(tD1 + (c & 1) * NS, x);
        mbar_wait(bar_v + 8 * (c & 1), (c >> 1) & 1, abort_flag);
        const unsigned char *vrow = sm + SM::kV + (c & 1) * SM::VI + t * 128;
#pragma unroll
        for (int ch = 0; ch < NH / 8; ch++) {
          const uint4 vv = *reinterpret_cast<const uint4 *>(vrow + (((c0 / 8 + ch) ^ (t & 7)) << 4));
          const __nv_bfloat162 *vb = reinterpret_cast<const __nv_bfloat162 *>(&vv);
          uint4 pk;
          __half2 *ph = reinterpret_cast<__half2 *>(&pk);
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const float2 vf = __bfloat1622float2(vb[i]);
            const float xa = x[ch * 8 + 2 * i];
            const float xb = x[ch * 8 + 2 * i + 1];
            ph[i] = __floats2half2_rn(beta_r * (vf.x - xa), beta_r * (vf.y - xb));
          }
          *reinterpret_cast<uint4 *>(sm + SM::kY + (c & 1) * SM::YI + mnmajor_chunk_off(t, c0 / 8 + ch, 64)) = pk;
        }
      }
      fence_proxy_async();
      fence_before_sync();
      named_bar(1, kChain);

      // ---- D2 = P1 Y; V buffer c & 1 is free: fetch chunk c + 2 into it ----
      if (tid == 0) {
        fence_after_sync();
        if (c + 2 < nchunks) issue_v(c + 2);
        const uint32_t sP = smem_addr(sm + SM::kP + s * SM::PI);
#pragma unroll
        for (int k0 = 0; k0 < C; k0 += 16) {  // K = C: rows of Y beyond C are zero
          const uint64_t bd = make_desc(sY + (c & 1) * SM::YI + (k0 >> 4) * 2048, 8 * 1024, 1024);
          const uint64_t ad = SM::COMPACT ? make_desc_sw64(sP + k0 * 2, 512) : make_desc(sP + k0 * 2, 16, 1024);
          mma_f16(tD2, ad, bd, idesc, k0 > 0 ? 1u : 0u);
        }
        mma_commit(bar_mma2);
        issue_o_intra(c);
      }
      mbar_wait(bar_mma2, c & 1, abort_flag);
      fence_after_sync();

      if (state_warp) {
        float d[NH];
        lane_half(tD2, d);
#pragma unroll
        for (int i = 0; i < NH; i++) s_reg[i] = fmaf(dec, s_reg[i], d[i]);
        write_state_image();
      }
      fence_proxy_async();
      fence_before_sync();
      named_bar(1, kChain);
    }
    if (nchunks > 0) {
      mbar_wait(bar_mma3, (nchunks - 1) & 1, abort_flag);
      fence_after_sync();
      if (query_warp) output_rows(nchunks - 1);
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
        // the prep kernel's gated fp16 [K~; Q~] image of this chunk
        bulk_g2s(smem_addr(sm + SM::kKQ + s * SM::KQ),
                 a.kq_images + ((size_t)(base + c) * a.HV + hv) * SM::KQ, SM::KQL, full);
        const unsigned char *src = reinterpret_cast<const unsigned char *>(a.tiles) +
                                   ((size_t)(base + c) * a.HV + hv) * kPrepImageBytes;
        bulk_g2s(smem_addr(sm + SM::kP + s * SM::PI), src, SM::PL, full);
      }
      float *raw = reinterpret_cast<float *>(sm + SM::kRaw + s * SM::NRAW * 4);
      // the chunk's per-channel decay (from the prep kernel) and beta
      if (pt < DK / 4)
        cp_async16(smem_addr(raw + 4 * pt), a.decays + ((size_t)(base + c) * a.HV + hv) * DK + 4 * pt, 16u);
      if (pt < C) {
        const bool in = pt < L;
        const long row = in ? (long)(t0 + pt) : (long)t0;
        cp_async4(smem_addr(raw + DK + pt), a.beta + row * a.HV + hv, in ? 4u : 0u);
      }
      cp_async_arrive_noinc(full);
    };

    // chunk c landed: its coefficients, then publish it
    auto finish = [&](int c) {
      const int s = c % NST;
      mbar_wait(bar_full + 8 * s, (c / NST) & 1, abort_flag);
      float *raw = reinterpret_cast<float *>(sm + SM::kRaw + s * SM::NRAW * 4);
      float *coef = reinterpret_cast<float *>(sm + SM::kCoef + s * SM::NCOEF * 4);
      if (pt < DK) coef[C + pt] = raw[pt];
      if (pt < C) coef[pt] = raw[DK + pt];
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

template <int C, int DK, int NST>
cudaError_t launch_one(const ScanArgs &a, const ScanMaps &maps, cudaStream_t stream) {
  using SM = ScanTcSmem<C, DK, NST>;
  auto kern = gdn_scan_tc_kernel<C, DK, NST>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (err != cudaSuccess) return err;
  const long blocks = (long)a.seq.n_seqs * a.HV * (a.dv / NS);
  if (blocks > 0x7fffffffL) return cudaErrorInvalidValue;
  kern<<<(unsigned)blocks, kThreads, SM::kBytes, stream>>>(a, maps);
  return cudaGetLastError();
}

template <int C, int DK>
cudaError_t dispatch_gate(const ScanArgs &a, const ScanMaps &m, int gate, cudaStream_t s) {
  // per-key gate only (the scalar gate runs gdn_scan_la.cu); two stages in flight
  if (!gate) return cudaErrorInvalidValue;
  return launch_one<C, DK, 2>(a, m, s);
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
