// gdn_transfer.cu -- composition of state transfers across sequence segments.
//
// Over any run of tokens the recurrence maps its entering state affinely:
// S_out = M S_in + S_seg, where S_seg is the state the run leaves from a zero
// start and M (dk x dk) is the state it leaves from the identity with all
// values zero (the value term of every update vanishes, so what remains is
// the product of the per-token maps (I - beta k k^T) diag(a)).  A long
// sequence split into segments that run on different GPUs therefore needs one
// exchange of (M, S_seg) per segment and one product per segment boundary
// (the sequence split with a state-transfer exchange of logismos issue #46,
// "Remaining work": independent positions, later continuation).  This kernel
// is that product, per (sequence, value head):
//     S_out = M S_in + S_seg          M [dk x dk], S_in, S_seg, S_out [dk x dv]
// in fp32, one thread per output element, the dk-long dot product in order.
#include <stdint.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

__global__ void __launch_bounds__(256) gdn_state_combine_kernel(TransferArgs a) {
  const long idx = blockIdx.x * 256L + threadIdx.x;
  const long per = (long)a.dk * a.dv;
  if (idx >= (long)a.n_states * per) return;
  const long h = idx / per;  // (sequence, value head)
  const int i = (int)((idx % per) / a.dv), j = (int)(idx % a.dv);
  const float *m = a.M + h * (long)a.dk * a.dk + (long)i * a.dk;
  const float *s = a.S_in + h * per + j;
  float acc = 0.f;
  for (int k = 0; k < a.dk; k++) acc = fmaf(__ldg(m + k), __ldg(s + (long)k * a.dv), acc);
  a.S_out[idx] = acc + a.S_seg[idx];
}

}  // namespace

cudaError_t launch_state_combine(const TransferArgs &a, cudaStream_t stream) {
  const long n = (long)a.n_states * a.dk * a.dv;
  if (n <= 0) return cudaSuccess;
  if ((n + 255) / 256 > 0x7fffffffL) return cudaErrorInvalidValue;
  gdn_state_combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
