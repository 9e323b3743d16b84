// gdn_internal.h -- declarations shared by the host API (gdn_api.cu) and the
// kernel translation units.  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// Bytes at the start of the workspace reserved for the device status word.
constexpr size_t kWorkspaceHeader = 256;
// Width of one dv slice handled by a scan CTA (fp32 path / bf16 path).
constexpr int kScanSlice = 32;
constexpr int kScanTcSlice = 64;
// The bf16 path's per-(chunk, value head) operand image written by the prep
// kernel: 192 rows x 64 fp16, K-major with the 128-byte swizzle
// (rows 0..127 = P1 = Kt^T T, rows 128..191 = Aqk T).
constexpr int kPrepImageRows = 192;
constexpr int kPrepImageBytes = kPrepImageRows * 128;
// At chunk 32 (per-key gate) its columns beyond C are never read: the image is
// written as 160 rows x 32 fp16 instead (K-major with the 64-byte swizzle; rows
// 0..127 = P1, rows 128..159 = Aqk T) in the first 10 KB of the same record.
constexpr int kPrepImage32Rows = 160;
constexpr int kPrepImage32Bytes = kPrepImage32Rows * 64;
// The scalar-gate bf16 path's image (one-chunk lookahead): 256 rows x 64 fp16,
// K-major with the 128-byte swizzle: rows 0..127 = P1 of the chunk, rows
// 128..191 = E = K_next P1 (the next chunk's keys times this chunk's P1; zero
// for a sequence's last chunk), rows 192..255 = Aqk T.
constexpr int kLaImageRows = 256;
constexpr int kLaImageBytes = kLaImageRows * 128;
// The same path's key/query image of one (chunk, q/k head): the A operand
// [K_next; Q] of the scan's state product, 128 rows of fp16 (next chunk's keys
// at 0..C-1, zero for a sequence's last chunk; this chunk's queries at
// 64..64+C-1), dk/64 panels of 128 x 128 bytes, K-major, 128-byte swizzle.
__host__ __device__ constexpr int kq_image_bytes(int dk) { return (dk / 64) * 16384; }

// Where packed sequence n starts: cu_seqlens[n], or n*T for plain batches.
// Sequence n owns the chunk slots [floor(start_n / C) + n, ...): one slot per
// chunk, injective over all sequences, fewer than floor(Ttot / C) + n_seqs.
struct SeqInfo {
  const int32_t *cu;  // device, or nullptr for a plain batch
  int n_seqs;         // sequences (B for a plain batch)
  int T;              // tokens per batch row (plain batch only)
  int Ttot;           // packed token count
};

struct PrepArgs {
  const void *q, *k;
  const float *g, *beta;
  SeqInfo seq;
  int H, HV;
  float scale;
  float *tiles;      // [n_slots][HV][2][C][C]: T = (I+A)^-1, then Aqk
  uint32_t *flags;   // device status word
  int n_slots;
  unsigned char *kq_images;  // bf16 scalar gate: [K_next; Q] image per (slot, hq);
                             // bf16 per-key gate: gated [K~; Q~] image per (slot, hv)
  float *decays;             // bf16 per-key gate: e^{b_last} per (slot, hv, key channel)
};

struct ScanArgs {
  const void *q, *k, *v;
  const float *g, *beta, *h0;
  void *o;
  float *hT;
  SeqInfo seq;
  int H, HV, dv;
  float scale;
  const float *tiles;
  uint32_t *flags;
  const unsigned char *kq_images;  // as PrepArgs::kq_images (read by the scan)
  const float *decays;             // as PrepArgs::decays
};

// The token-serial form (gdn_recurrent.cu): state in registers, one token at
// a time; hT may be h0 itself.
struct RecurrentArgs {
  const void *q, *k, *v;
  const float *g, *beta, *h0;
  void *o;
  float *hT;
  SeqInfo seq;
  int H, HV, dv;
  float scale;
  uint32_t *flags;  // device status word, or nullptr
};

// The operations either side of the recurrence (gdn_prepost.cu).
struct ConvArgs {
  const void *x;
  const float *w, *bias, *h0;  // w [D][W]; bias [D] or nullptr; h0 [N][D][W-1] or nullptr
  void *y;
  float *hT;                   // [N][D][W-1] or nullptr; may be h0 itself
  SeqInfo seq;
  int D;
  uint32_t *flags;             // device status word, or nullptr
  int tile0 = 0;               // first token tile of this launch (set by the launcher)
};
struct RowNormArgs {
  const void *x, *z;           // z: gate rows (gated RMS norm only), or nullptr
  const float *weight;         // [dim] (gated RMS norm only)
  void *y;
  long rows;
  float eps;
};

// Composition of a segment's state transfer (gdn_transfer.cu):
// S_out = M S_in + S_seg per (state, value head); n_states = sequences x heads.
struct TransferArgs {
  const float *M, *S_in, *S_seg;
  float *S_out;
  long n_states;
  int dk, dv;
};

// Status-word bits (same values as GDN_FLAG_* in include/gdn.h).
constexpr uint32_t kFlagPositiveGate = 1u << 0;
constexpr uint32_t kFlagNonfinite = 1u << 1;
constexpr uint32_t kFlagBadSeqlens = 1u << 2;
constexpr uint32_t kFlagTimeout = 1u << 3;
constexpr uint32_t kFlagLaunchConfig = 1u << 4;

// Launchers; return cudaErrorInvalidValue for an uncompiled combination.
// dtype: 0 = fp32, 1 = bf16.  gate: 0 = scalar (GDN), 1 = per key (KDA).
cudaError_t launch_prep(const PrepArgs &a, int chunk, int dk, int dtype,
                        int gate, cudaStream_t stream);
cudaError_t launch_scan(const ScanArgs &a, int chunk, int dk, int dtype,
                        int gate, cudaStream_t stream);
// TMA descriptors of the bf16 path's scan: q, k as [Ttot][H][dk] and v as
// [Ttot][HV][dv], boxes of 64 columns x 1 head x C tokens, 128-byte swizzle.
struct ScanMaps {
  CUtensorMap q, k, v;
  CUtensorMap g;  // per-key gates (fp32 [Ttot][HV][dk], box 64 x 1 x chunk); zero otherwise
};
// Encode the maps (host); `g_per_key` null for the scalar gate.  False when
// the driver refuses.
bool make_scan_maps(ScanMaps &m, const void *q, const void *k, const void *v,
                    const float *g_per_key, int Ttot, int H, int HV, int dk, int dv, int chunk);

// bf16 per-key-gate path: prep writing fp16 operand images, tcgen05 scan
// consuming them
cudaError_t launch_prep_tc(const PrepArgs &a, int chunk, int dk, int gate,
                           cudaStream_t stream);
// bf16 per-key-gate prep at chunk 32 (gdn_prep_kda.cu): TMA tiles, the
// factored A / Aqk product on tcgen05; same outputs as launch_prep_tc
cudaError_t launch_prep_kda(const PrepArgs &a, const ScanMaps &maps, int dk, cudaStream_t stream);
cudaError_t launch_scan_tc(const ScanArgs &a, const ScanMaps &maps, int chunk, int dk,
                           int gate, cudaStream_t stream);
// bf16 scalar-gate path: prep on tensor memory writing the lookahead image,
// and the lookahead scan consuming it
// (n_slots >= 0: only the first n_slots chunk slots; ready != nullptr: each
// unit's flag in ready[slot * H + hq] is set once its images are complete)
cudaError_t launch_prep_tmem(const PrepArgs &a, const ScanMaps &maps, int chunk, int dk,
                             cudaStream_t stream, int n_slots = -1, int *ready = nullptr);
cudaError_t launch_scan_la(const ScanArgs &a, const ScanMaps &maps, int chunk, int dk,
                           cudaStream_t stream);
// the same two computations in one cooperative launch, the scan loading each
// prep image once the prep has set its (chunk slot, q/k head) flag in
// `ready` (n_slots x H ints, zeroed beforehand); the prep warpgroups take the
// units from slot `head_slots` on (the earlier ones come from a prep launch
// over the first head_slots slots, enqueued just before; head_slots < 0:
// chosen from the problem's shape);
// cudaErrorCooperativeLaunchTooLarge when the scan's blocks leave no SM for
// the prep
cudaError_t launch_lockstep(const PrepArgs &pa, const ScanArgs &sa, const ScanMaps &maps,
                            int *ready, int head_slots, int chunk, int dk, cudaStream_t stream);
// causal depthwise convolution (width 1..4, D a multiple of 8; activation 0 =
// none, 1 = SiLU) and the row norms (kind 0 = L2, 1 = gated RMS; dim 64, 128
// or 256)
cudaError_t launch_conv1d(const ConvArgs &a, int width, int activation, int dtype,
                          cudaStream_t stream);
cudaError_t launch_rownorm(const RowNormArgs &a, int dim, int kind, int dtype,
                           cudaStream_t stream);
// S_out = M S_in + S_seg, per state
cudaError_t launch_state_combine(const TransferArgs &a, cudaStream_t stream);
// token-serial form; dv a multiple of 32
cudaError_t launch_recurrent(const RecurrentArgs &a, int dk, int dtype, int gate,
                             cudaStream_t stream);

}  // namespace gdn
