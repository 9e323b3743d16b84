// gdn_noalloc.cu -- gdn_chunk_fwd for callers that cannot allocate device
// memory.
//
// Some callers are not allowed to call cudaMalloc: components embedded in a
// host framework that owns every byte of device memory and gives plug-ins none
// of their own, or latency-critical loops where an allocation could stall the
// device.  gdn_chunk_fwd needs a workspace (the prep kernel's per-chunk T and
// Aqk tiles plus the status word), which such a caller has no way to provide.
// This entry point runs the same two kernels with the workspace taken from a
// fixed device array of kStaticScratchBytes that lives in this library: it is
// reserved on every GPU that loads the library, for as long as the process
// lives.  Nothing here allocates: no cudaMalloc, no cudaFree, no allocating
// library routine.
//
// Sharing rules: every call on a device uses the same array.  Calls that
// overlap on the GPU (on different streams, or from different threads without
// ordering) race on it and corrupt each other's results; serialise them.  The
// array keeps the last call's contents.  Nothing in it must start at zero
// except the status word, which every call clears itself before its kernels
// run; every tile the scan kernel reads is written by the prep kernel of the
// same call first.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gdn.h"

namespace {

// Maximum workspace of one call: 64 MiB (e.g. 4096 tokens x 16 value heads at
// chunk 64, or 16384 tokens x 4 value heads).
constexpr size_t kStaticScratchBytes = size_t(64) << 20;

// Device-side scratch.  In host code this name is only a stand-in for the
// symbol, not a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char gdn_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).  nullptr on failure.
void *scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, gdn_static_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" gdn_status gdn_chunk_fwd_noalloc(
    const void *q, const void *k, const void *v, const float *g, const float *beta,
    const float *h0, void *o, float *hT, const int32_t *cu_seqlens, int n_seqs, int B,
    int T, int H, int HV, int dk, int dv, int chunk, float scale, int gate_mode,
    int dtype, gdn_stream_t stream) {
  // workspace this request needs; 0 means gdn_chunk_fwd refuses the request,
  // and it then returns the precise reason itself below
  const size_t need = gdn_chunk_fwd_workspace_bytes(B, T, H, HV, dk, dv, chunk, gate_mode,
                                                    cu_seqlens ? n_seqs : B, dtype);
  if (need > kStaticScratchBytes) return GDN_ERR_WORKSPACE;
  void *scratch = scratch_on_current_device();
  if (!scratch) return GDN_ERR_CUDA;
  return gdn_chunk_fwd(q, k, v, g, beta, h0, o, hT, cu_seqlens, n_seqs, B, T, H, HV, dk,
                       dv, chunk, scale, gate_mode, dtype, scratch, kStaticScratchBytes,
                       stream);
}
