// gdn_api.cu -- host side of the C ABI declared in include/gdn.h: argument
// validation, workspace sizing and the two launches (prep, then scan) on the
// caller's stream, and the one launch of the token-serial form.  Unsupported
// requests are refused explicitly, before anything is enqueued (logismos
// issue #46, "Acceptance": unsupported inputs fail explicitly).
#include <cuda_runtime.h>
#include <stdint.h>

#include <cudaTypedefs.h>

#include <cmath>
#include <cstddef>
#include <cstring>
#include <mutex>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 tensor [d2][d1][d0] (d0 contiguous), box {b0, 1, b2}, 128-byte swizzle
bool map3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
           uint32_t b2) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {b0, 1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 tensor [d2][d1][d0] (d0 contiguous), box {b0, 1, b2}, no swizzle
bool map3d_f32(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint32_t b0, uint32_t b2) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 4, d0 * d1 * 4};
  const cuuint32_t box[3] = {b0, 1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_scan_maps(ScanMaps &m, const void *q, const void *k, const void *v,
                    const float *g_per_key, int Ttot, int H, int HV, int dk, int dv, int chunk) {
  std::memset(&m, 0, sizeof(m));
  if (Ttot <= 0) return true;  // nothing will be loaded
  if (!encode_fn()) return false;
  return map3d(&m.q, q, dk, H, Ttot, 64, chunk) && map3d(&m.k, k, dk, H, Ttot, 64, chunk) &&
         map3d(&m.v, v, dv, HV, Ttot, kScanTcSlice, chunk) &&
         (!g_per_key || map3d_f32(&m.g, g_per_key, dk, HV, Ttot, 64, chunk));
}

}  // namespace gdn

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

struct Plan {
  int n_states;   // B, or n_seqs when packed
  long Ttot;      // packed token count
  long n_slots;   // chunk slots of the workspace
  size_t tile_bytes;
  size_t kq_bytes;
  size_t decay_bytes;
  size_t ready_bytes;
  size_t ws_bytes;
};

// Shape checks shared by the workspace query and the call.  Returns GDN_OK
// and fills `p`, or the status the call must return.
gdn_status plan(int B, int T, int H, int HV, int dk, int dv, int chunk,
                int gate_mode, int n_seqs, int dtype, bool packed, Plan &p) {
  if (B <= 0 || T < 0 || H <= 0 || HV <= 0 || dk <= 0 || dv <= 0 || chunk <= 0)
    return GDN_ERR_INVALID_ARG;
  if (HV % H != 0 || HV > 65535) return GDN_ERR_INVALID_ARG;
  if (gate_mode != GDN_GATE_SCALAR && gate_mode != GDN_GATE_PER_KEY) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (packed) {
    if (B != 1 || n_seqs <= 0) return GDN_ERR_INVALID_ARG;
    p.n_states = n_seqs;
  } else {
    if (n_seqs != 0 && n_seqs != B) return GDN_ERR_INVALID_ARG;
    p.n_states = B;
  }
  if (!(dk == 64 || dk == 128) || !(dv == 64 || dv == 128)) return GDN_ERR_UNSUPPORTED;
  if (!(chunk == 32 || chunk == 64)) return GDN_ERR_UNSUPPORTED;
  p.Ttot = (long)B * T;
  if (p.Ttot > INT32_MAX - 2L * chunk) return GDN_ERR_UNSUPPORTED;
  p.n_slots = p.Ttot / chunk + p.n_states;
  if (p.n_slots > INT32_MAX) return GDN_ERR_UNSUPPORTED;
  // fp32 inputs: T and Aqk as fp32 C x C tiles; bf16 inputs: one fp16 operand
  // image per (chunk, value head), [P1; E; AqkT] for the scalar gate and
  // [P1; AqkT] for the per-key gate
  size_t per = 2u * (size_t)chunk * (size_t)chunk * sizeof(float);
  if (dtype == GDN_BF16)
    per = gate_mode == GDN_GATE_SCALAR ? (size_t)gdn::kLaImageBytes : (size_t)gdn::kPrepImageBytes;
  p.tile_bytes = (size_t)p.n_slots * (size_t)HV * per;
  // bf16: the prep kernel also publishes key/query images, [K_next; Q] per
  // (slot, q/k head) for the scalar gate, gated [K~; Q~] per (slot, value
  // head) for the per-key gate, which also gets each chunk's per-channel decay
  p.kq_bytes = 0;
  p.decay_bytes = 0;
  if (dtype == GDN_BF16) {
    const size_t heads = gate_mode == GDN_GATE_SCALAR ? (size_t)H : (size_t)HV;
    p.kq_bytes = (size_t)p.n_slots * heads * (size_t)gdn::kq_image_bytes(dk);
    if (gate_mode == GDN_GATE_PER_KEY) p.decay_bytes = (size_t)p.n_slots * HV * dk * sizeof(float);
  }
  // bf16 scalar gate: one ready flag per (slot, q/k head) for the lockstep
  // launch, 256-byte padded
  p.ready_bytes = 0;
  if (dtype == GDN_BF16 && gate_mode == GDN_GATE_SCALAR)
    p.ready_bytes = ((size_t)p.n_slots * (size_t)H * sizeof(int) + 255) / 256 * 256;
  p.ws_bytes = gdn::kWorkspaceHeader + p.tile_bytes + p.kq_bytes + p.decay_bytes + p.ready_bytes;
  return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_version(void) { return 100; }

const char *gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    default: return "GDN_ERR_UNKNOWN";
  }
}

size_t gdn_chunk_fwd_workspace_bytes(int B, int T, int H, int HV, int dk, int dv,
                                     int chunk, int gate_mode, int n_seqs, int dtype) {
  Plan p;
  // a packed request is one with B == 1 and n_seqs > 1, or n_seqs given with B == 1;
  // the size only depends on the number of states, so both readings agree
  const bool packed = (B == 1 && n_seqs > 1);
  if (plan(B, T, H, HV, dk, dv, chunk, gate_mode, n_seqs, dtype, packed, p) != GDN_OK) return 0;
  return p.ws_bytes;
}

}  // extern "C"

namespace {

enum Stage { kPrep = 1, kScan = 2, kBoth = 3, kLockstep = 4 };

gdn_status run(int stages, const void *q, const void *k, const void *v, const float *g,
               const float *beta, const float *h0, void *o, float *hT,
               const int32_t *cu_seqlens, int n_seqs, int B, int T, int H, int HV, int dk,
               int dv, int chunk, float scale, int gate_mode, int dtype, void *workspace,
               size_t workspace_bytes, gdn_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const bool packed = cu_seqlens != nullptr;
  Plan p;
  gdn_status st = plan(B, T, H, HV, dk, dv, chunk, gate_mode, n_seqs, dtype, packed, p);
  if (st != GDN_OK) return st;
  if (!std::isfinite(scale)) return GDN_ERR_INVALID_ARG;
  // the lockstep launch exists for the bf16 scalar-gate path only
  if (stages == kLockstep && !(dtype == GDN_BF16 && gate_mode == GDN_GATE_SCALAR))
    return GDN_ERR_UNSUPPORTED;

  // pointers: required ones non-null (token data may be absent when there are
  // no tokens), all 16-byte aligned
  if (p.Ttot > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, h0, o, hT, cu_seqlens, workspace};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < p.ws_bytes) return GDN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_INVALID_ARG;

  // aliasing: hT vs h0; o and hT vs every input; workspace vs everything
  const size_t es = dtype == GDN_BF16 ? 2 : 4;
  const size_t n_qk = (size_t)p.Ttot * H * dk * es;
  const size_t n_vo = (size_t)p.Ttot * HV * dv * es;
  const size_t n_g = (size_t)p.Ttot * HV * (gate_mode == GDN_GATE_PER_KEY ? dk : 1) * 4;
  const size_t n_b = (size_t)p.Ttot * HV * 4;
  const size_t n_h = (size_t)p.n_states * HV * dk * dv * 4;
  if (overlap(hT, n_h, h0, n_h)) return GDN_ERR_INVALID_ARG;
  const void *ins[] = {q, k, v, g, beta, h0};
  const size_t in_n[] = {n_qk, n_qk, n_vo, n_g, n_b, n_h};
  for (int i = 0; i < 6; i++) {
    if (overlap(o, n_vo, ins[i], in_n[i])) return GDN_ERR_INVALID_ARG;
    if (overlap(hT, n_h, ins[i], in_n[i])) return GDN_ERR_INVALID_ARG;
    if (overlap(workspace, p.ws_bytes, ins[i], in_n[i])) return GDN_ERR_INVALID_ARG;
  }
  if (overlap(o, n_vo, hT, n_h) || overlap(workspace, p.ws_bytes, o, n_vo) ||
      overlap(workspace, p.ws_bytes, hT, n_h))
    return GDN_ERR_INVALID_ARG;

  uint32_t *flags = static_cast<uint32_t *>(workspace);
  gdn::SeqInfo seq;
  seq.cu = cu_seqlens;
  seq.n_seqs = p.n_states;
  seq.T = T;
  seq.Ttot = (int)p.Ttot;
  float *tiles = reinterpret_cast<float *>(static_cast<char *>(workspace) + gdn::kWorkspaceHeader);
  unsigned char *kq_images =
      p.kq_bytes ? static_cast<unsigned char *>(workspace) + gdn::kWorkspaceHeader + p.tile_bytes
                 : nullptr;
  float *decays = p.decay_bytes ? reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                            gdn::kWorkspaceHeader + p.tile_bytes +
                                                            p.kq_bytes)
                                : nullptr;
  int *ready = p.ready_bytes ? reinterpret_cast<int *>(static_cast<char *>(workspace) +
                                                       gdn::kWorkspaceHeader + p.tile_bytes +
                                                       p.kq_bytes + p.decay_bytes)
                             : nullptr;

  gdn::ScanMaps maps;
  if (dtype == GDN_BF16 &&
      !gdn::make_scan_maps(maps, q, k, v, gate_mode == GDN_GATE_PER_KEY ? g : nullptr,
                           (int)p.Ttot, H, HV, dk, dv, chunk))
    return GDN_ERR_CUDA;
  if (stages == kLockstep) {
    if (cudaMemsetAsync(flags, 0, sizeof(uint32_t), stream) != cudaSuccess) return GDN_ERR_CUDA;
    if (p.Ttot == 0 && !hT) return GDN_OK;
    if (cudaMemsetAsync(ready, 0, p.ready_bytes, stream) != cudaSuccess) return GDN_ERR_CUDA;
    gdn::PrepArgs pa;
    pa.q = q; pa.k = k; pa.g = g; pa.beta = beta;
    pa.seq = seq; pa.H = H; pa.HV = HV; pa.scale = scale;
    pa.tiles = tiles; pa.flags = flags; pa.n_slots = (int)p.n_slots;
    pa.kq_images = kq_images;
    pa.decays = decays;
    gdn::ScanArgs sa;
    sa.q = q; sa.k = k; sa.v = v; sa.g = g; sa.beta = beta; sa.h0 = h0;
    sa.o = o; sa.hT = hT; sa.seq = seq; sa.H = H; sa.HV = HV; sa.dv = dv;
    sa.scale = scale; sa.tiles = tiles; sa.flags = flags; sa.kq_images = kq_images;
    sa.decays = decays;
    // the prep's head start is chosen by the launcher
    const cudaError_t e = gdn::launch_lockstep(pa, sa, maps, ready, -1, chunk, dk, stream);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
      (void)cudaGetLastError();
      return GDN_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  }
  if (stages & kPrep) {
    if (cudaMemsetAsync(flags, 0, sizeof(uint32_t), stream) != cudaSuccess) return GDN_ERR_CUDA;
    if (p.Ttot > 0) {
      gdn::PrepArgs pa;
      pa.q = q; pa.k = k; pa.g = g; pa.beta = beta;
      pa.seq = seq; pa.H = H; pa.HV = HV; pa.scale = scale;
      pa.tiles = tiles; pa.flags = flags; pa.n_slots = (int)p.n_slots;
      pa.kq_images = kq_images;
      pa.decays = decays;
      cudaError_t e;
      if (dtype == GDN_BF16 && gate_mode == GDN_GATE_SCALAR)
        e = gdn::launch_prep_tmem(pa, maps, chunk, dk, stream);
      else if (dtype == GDN_BF16 && chunk == 32)
        e = gdn::launch_prep_kda(pa, maps, dk, stream);
      else if (dtype == GDN_BF16)
        e = gdn::launch_prep_tc(pa, chunk, dk, gate_mode, stream);
      else
        e = gdn::launch_prep(pa, chunk, dk, dtype, gate_mode, stream);
      if (e != cudaSuccess) return GDN_ERR_CUDA;
    }
  }
  if (stages & kScan) {
    gdn::ScanArgs sa;
    sa.q = q; sa.k = k; sa.v = v; sa.g = g; sa.beta = beta; sa.h0 = h0;
    sa.o = o; sa.hT = hT; sa.seq = seq; sa.H = H; sa.HV = HV; sa.dv = dv;
    sa.scale = scale; sa.tiles = tiles; sa.flags = flags; sa.kq_images = kq_images;
    sa.decays = decays;
    cudaError_t e;
    if (dtype == GDN_BF16 && gate_mode == GDN_GATE_SCALAR)
      e = gdn::launch_scan_la(sa, maps, chunk, dk, stream);
    else if (dtype == GDN_BF16)
      e = gdn::launch_scan_tc(sa, maps, chunk, dk, gate_mode, stream);
    else
      e = gdn::launch_scan(sa, chunk, dk, dtype, gate_mode, stream);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
  }
  return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, const float *h0, void *o, float *hT,
                         const int32_t *cu_seqlens, int n_seqs, int B, int T, int H,
                         int HV, int dk, int dv, int chunk, float scale, int gate_mode,
                         int dtype, void *workspace, size_t workspace_bytes,
                         gdn_stream_t stream) {
  return run(kBoth, q, k, v, g, beta, h0, o, hT, cu_seqlens, n_seqs, B, T, H, HV, dk, dv,
             chunk, scale, gate_mode, dtype, workspace, workspace_bytes, stream);
}

gdn_status gdn_chunk_fwd_lockstep(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, const float *h0, void *o, float *hT,
                                  const int32_t *cu_seqlens, int n_seqs, int B, int T, int H,
                                  int HV, int dk, int dv, int chunk, float scale, int gate_mode,
                                  int dtype, void *workspace, size_t workspace_bytes,
                                  gdn_stream_t stream) {
  return run(kLockstep, q, k, v, g, beta, h0, o, hT, cu_seqlens, n_seqs, B, T, H, HV, dk, dv,
             chunk, scale, gate_mode, dtype, workspace, workspace_bytes, stream);
}

gdn_status gdn_chunk_fwd_prep(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, const float *h0, void *o, float *hT,
                              const int32_t *cu_seqlens, int n_seqs, int B, int T, int H,
                              int HV, int dk, int dv, int chunk, float scale, int gate_mode,
                              int dtype, void *workspace, size_t workspace_bytes,
                              gdn_stream_t stream) {
  return run(kPrep, q, k, v, g, beta, h0, o, hT, cu_seqlens, n_seqs, B, T, H, HV, dk, dv,
             chunk, scale, gate_mode, dtype, workspace, workspace_bytes, stream);
}

gdn_status gdn_chunk_fwd_scan(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, const float *h0, void *o, float *hT,
                              const int32_t *cu_seqlens, int n_seqs, int B, int T, int H,
                              int HV, int dk, int dv, int chunk, float scale, int gate_mode,
                              int dtype, void *workspace, size_t workspace_bytes,
                              gdn_stream_t stream) {
  return run(kScan, q, k, v, g, beta, h0, o, hT, cu_seqlens, n_seqs, B, T, H, HV, dk, dv,
             chunk, scale, gate_mode, dtype, workspace, workspace_bytes, stream);
}

gdn_status gdn_recurrent_fwd(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const float *h0, void *o, float *hT,
                             const int32_t *cu_seqlens, int n_seqs, int B, int T, int H,
                             int HV, int dk, int dv, float scale, int gate_mode, int dtype,
                             uint32_t *flags, gdn_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (B <= 0 || T < 0 || H <= 0 || HV <= 0 || dk <= 0 || dv <= 0) return GDN_ERR_INVALID_ARG;
  if (HV % H != 0 || HV > 65535) return GDN_ERR_INVALID_ARG;
  if (gate_mode != GDN_GATE_SCALAR && gate_mode != GDN_GATE_PER_KEY) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GDN_ERR_INVALID_ARG;
  const bool packed = cu_seqlens != nullptr;
  int n_states;
  if (packed) {
    if (B != 1 || n_seqs <= 0) return GDN_ERR_INVALID_ARG;
    n_states = n_seqs;
  } else {
    if (n_seqs != 0 && n_seqs != B) return GDN_ERR_INVALID_ARG;
    n_states = B;
  }
  if (!(dk == 64 || dk == 128) || dv % 32 != 0 || dv > 1024) return GDN_ERR_UNSUPPORTED;
  const long Ttot = (long)B * T;
  if (Ttot > INT32_MAX) return GDN_ERR_UNSUPPORTED;

  if (Ttot > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, h0, o, hT, cu_seqlens};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  if (flags && (reinterpret_cast<uintptr_t>(flags) & 3u) != 0) return GDN_ERR_INVALID_ARG;

  // aliasing: hT may be h0 itself (an in-place state update), not a part of it;
  // o, hT and the status word overlap no input and no other output
  const size_t es = dtype == GDN_BF16 ? 2 : 4;
  const size_t n_qk = (size_t)Ttot * H * dk * es;
  const size_t n_vo = (size_t)Ttot * HV * dv * es;
  const size_t n_g = (size_t)Ttot * HV * (gate_mode == GDN_GATE_PER_KEY ? dk : 1) * 4;
  const size_t n_b = (size_t)Ttot * HV * 4;
  const size_t n_h = (size_t)n_states * HV * dk * dv * 4;
  const size_t n_cu = packed ? ((size_t)n_seqs + 1) * 4 : 0;
  if (hT != h0 && overlap(hT, n_h, h0, n_h)) return GDN_ERR_INVALID_ARG;
  const void *ins[] = {q, k, v, g, beta, cu_seqlens};
  const size_t in_n[] = {n_qk, n_qk, n_vo, n_g, n_b, n_cu};
  for (int i = 0; i < 6; i++) {
    if (overlap(o, n_vo, ins[i], in_n[i]) || overlap(hT, n_h, ins[i], in_n[i]) ||
        overlap(flags, 4, ins[i], in_n[i]))
      return GDN_ERR_INVALID_ARG;
  }
  if (overlap(o, n_vo, h0, n_h) || overlap(o, n_vo, hT, n_h) || overlap(flags, 4, o, n_vo) ||
      overlap(flags, 4, h0, n_h) || overlap(flags, 4, hT, n_h))
    return GDN_ERR_INVALID_ARG;

  if (flags && cudaMemsetAsync(flags, 0, sizeof(uint32_t), stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  gdn::RecurrentArgs ra;
  ra.q = q; ra.k = k; ra.v = v; ra.g = g; ra.beta = beta; ra.h0 = h0;
  ra.o = o; ra.hT = hT;
  ra.seq.cu = cu_seqlens;
  ra.seq.n_seqs = n_states;
  ra.seq.T = T;
  ra.seq.Ttot = (int)Ttot;
  ra.H = H; ra.HV = HV; ra.dv = dv; ra.scale = scale; ra.flags = flags;
  if (gdn::launch_recurrent(ra, dk, dtype, gate_mode, stream) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}

gdn_status gdn_causal_conv1d_fwd(const void *x, const float *w, const float *bias,
                                 const float *h0, void *y, float *hT,
                                 const int32_t *cu_seqlens, int n_seqs, int B, int T, int D,
                                 int width, int activation, int dtype, uint32_t *flags,
                                 gdn_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (B <= 0 || T < 0 || D <= 0 || width <= 0) return GDN_ERR_INVALID_ARG;
  if (activation != GDN_ACT_NONE && activation != GDN_ACT_SILU) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  const bool packed = cu_seqlens != nullptr;
  int n_states;
  if (packed) {
    if (B != 1 || n_seqs <= 0) return GDN_ERR_INVALID_ARG;
    n_states = n_seqs;
  } else {
    if (n_seqs != 0 && n_seqs != B) return GDN_ERR_INVALID_ARG;
    n_states = B;
  }
  if (width > 4 || D % 8 != 0) return GDN_ERR_UNSUPPORTED;
  const long Ttot = (long)B * T;
  if (Ttot > INT32_MAX || (long)n_states * D > INT32_MAX) return GDN_ERR_UNSUPPORTED;
  if (!w || (Ttot > 0 && (!x || !y))) return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {x, w, bias, h0, y, hT, cu_seqlens};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  if (flags && (reinterpret_cast<uintptr_t>(flags) & 3u) != 0) return GDN_ERR_INVALID_ARG;
  const size_t es = dtype == GDN_BF16 ? 2 : 4;
  const size_t n_x = (size_t)Ttot * D * es, n_w = (size_t)D * width * 4, n_b = (size_t)D * 4;
  const size_t n_h = (size_t)n_states * D * (width - 1) * 4;
  const size_t n_cu = packed ? ((size_t)n_seqs + 1) * 4 : 0;
  if (hT != h0 && overlap(hT, n_h, h0, n_h)) return GDN_ERR_INVALID_ARG;
  const void *ins[] = {x, w, bias, cu_seqlens};
  const size_t in_n[] = {n_x, n_w, n_b, n_cu};
  for (int i = 0; i < 4; i++)
    if (overlap(y, n_x, ins[i], in_n[i]) || overlap(hT, n_h, ins[i], in_n[i]) ||
        overlap(flags, 4, ins[i], in_n[i]))
      return GDN_ERR_INVALID_ARG;
  if (overlap(y, n_x, h0, n_h) || overlap(y, n_x, hT, n_h) || overlap(flags, 4, y, n_x) ||
      overlap(flags, 4, h0, n_h) || overlap(flags, 4, hT, n_h))
    return GDN_ERR_INVALID_ARG;

  if (flags && cudaMemsetAsync(flags, 0, sizeof(uint32_t), stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  gdn::ConvArgs ca;
  ca.x = x; ca.w = w; ca.bias = bias; ca.h0 = h0; ca.y = y; ca.hT = hT;
  ca.seq.cu = cu_seqlens;
  ca.seq.n_seqs = n_states;
  ca.seq.T = T;
  ca.seq.Ttot = (int)Ttot;
  ca.D = D;
  ca.flags = flags;
  if (gdn::launch_conv1d(ca, width, activation, dtype, stream) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}

static gdn_status rownorm(int kind, const void *x, const void *z, const float *weight, void *y,
                          int64_t rows, int dim, float eps, int dtype, gdn_stream_t stream_) {
  if (rows < 0 || dim <= 0 || !(eps >= 0.f) || !std::isfinite(eps)) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (!(dim == 64 || dim == 128 || dim == 256)) return GDN_ERR_UNSUPPORTED;
  if (rows > 0 && (!x || !y)) return GDN_ERR_INVALID_ARG;
  if (kind == 1 && !weight) return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {x, z, weight, y};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  const size_t es = dtype == GDN_BF16 ? 2 : 4;
  const size_t n = (size_t)rows * dim * es;
  // y may be x itself (in place); any other overlap is refused
  if (y != x && overlap(y, n, x, n)) return GDN_ERR_INVALID_ARG;
  if (overlap(y, n, z, n) || overlap(y, n, weight, (size_t)dim * 4)) return GDN_ERR_INVALID_ARG;
  gdn::RowNormArgs ra;
  ra.x = x; ra.z = z; ra.weight = weight; ra.y = y; ra.rows = (long)rows; ra.eps = eps;
  if (gdn::launch_rownorm(ra, dim, kind, dtype, reinterpret_cast<cudaStream_t>(stream_)) !=
      cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

gdn_status gdn_l2norm_fwd(const void *x, void *y, int64_t rows, int dim, float eps, int dtype,
                          gdn_stream_t stream) {
  return rownorm(0, x, nullptr, nullptr, y, rows, dim, eps, dtype, stream);
}

gdn_status gdn_rmsnorm_gated_fwd(const void *x, const void *z, const float *weight, void *y,
                                 int64_t rows, int dim, float eps, int dtype,
                                 gdn_stream_t stream) {
  return rownorm(1, x, z, weight, y, rows, dim, eps, dtype, stream);
}

gdn_status gdn_state_combine(const float *M, const float *S_in, const float *S_seg,
                             float *S_out, int n_seqs, int HV, int dk, int dv,
                             gdn_stream_t stream) {
  if (n_seqs < 0 || HV <= 0 || dk <= 0 || dv <= 0) return GDN_ERR_INVALID_ARG;
  if (dk > 1024 || dv > 1024) return GDN_ERR_UNSUPPORTED;
  const long n_states = (long)n_seqs * HV;
  if (n_states > 0 && (!M || !S_in || !S_seg || !S_out)) return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {M, S_in, S_seg, S_out};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  const size_t n_m = (size_t)n_states * dk * dk * 4, n_s = (size_t)n_states * dk * dv * 4;
  // S_out may be S_seg itself; it overlaps nothing else
  if (overlap(S_out, n_s, M, n_m) || overlap(S_out, n_s, S_in, n_s)) return GDN_ERR_INVALID_ARG;
  if (S_out != S_seg && overlap(S_out, n_s, S_seg, n_s)) return GDN_ERR_INVALID_ARG;
  gdn::TransferArgs ta;
  ta.M = M; ta.S_in = S_in; ta.S_seg = S_seg; ta.S_out = S_out;
  ta.n_states = n_states; ta.dk = dk; ta.dv = dv;
  if (gdn::launch_state_combine(ta, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

gdn_status gdn_read_device_flags(const void *workspace, uint32_t *flags_out,
                                 gdn_stream_t stream_) {
  if (!workspace || !flags_out) return GDN_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
  *flags_out = v;
  return GDN_OK;
}

}  // extern "C"
