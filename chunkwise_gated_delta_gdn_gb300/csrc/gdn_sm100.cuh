// gdn_sm100.cuh -- hand-written PTX for the 5th-generation tensor cores of
// sm_100-class GPUs (GB300 = sm_103a): shared-memory matrix descriptors,
// tcgen05.mma (kind::f16, fp32 accumulation in tensor memory), commit to an
// mbarrier, tensor-memory allocation and loads, bulk copies, and mbarrier
// waits that give up after a clock budget instead of spinning forever.
//
// Operand images in shared memory use the 128-byte swizzle:
//  * K-major (rows of the M or N dimension, K contiguous): 128-byte rows of 64
//    16-bit elements, 8-row atoms of 1024 bytes, atoms stacked along M/N
//    (stride-byte-offset 1024); a K extent above 64 lives in further
//    "panels" of rows x 128 bytes.  A K step of 16 advances the start
//    address by 32 bytes inside the row.
//  * MN-major (rows of the K dimension, M/N contiguous): 128-byte rows of 64
//    16-bit M/N elements, 8 K-rows per 1024-byte atom; K groups stacked with
//    stride-byte-offset 1024, further 64-element M/N atoms at the
//    leading-byte-offset.  A K step of 16 advances the start by 2048 bytes.
// In both, the 16-byte chunk index inside a row is XORed with (row % 8).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace gdn {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of 16-bit element (row, k) in a K-major image of `rows` rows
__device__ __forceinline__ uint32_t kmajor_off(int row, int k, int rows) {
  const int panel = k >> 6, kk = k & 63;
  return panel * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
         ((((kk * 2) >> 4) ^ (row & 7)) << 4) + ((kk * 2) & 15);
}

// byte offset of the 16-byte chunk `chunk` (8 elements) of K-row `k` in an
// MN-major image with `krows` K-rows (MN atom stride krows/8 * 1024 bytes)
__device__ __forceinline__ uint32_t mnmajor_chunk_off(int k, int chunk, int krows) {
  const int atom = chunk >> 3, cc = chunk & 7;
  return atom * (krows >> 3) * 1024 + (k >> 3) * 1024 + (k & 7) * 128 + ((cc ^ (k & 7)) << 4);
}

__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of sm_100-class tensor cores
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// The same for K-major images with 64-byte rows (32 16-bit elements) in the
// 64-byte swizzle: 8-row atoms of 512 bytes, the 16-byte chunk index inside a
// row XORed with (row / 2) % 4.
__device__ __forceinline__ uint32_t kmajor64_off(int row, int k) {
  return row * 64 + (((((k * 2) >> 4) ^ (row >> 1)) & 3) << 4) + ((k * 2) & 15);
}
__device__ __forceinline__ uint64_t make_desc_sw64(uint32_t saddr, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;  // leading-byte offset (unused by swizzled K-major operands)
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;  // 64-byte swizzle
  return d;
}

// instruction descriptor: fp16 A and B, fp32 D, M x N, operand majorness
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// the same with bf16 A and B (both operands of one product share a type)
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return idesc_f16(M, N, a_mn, b_mn) | (1u << 7) | (1u << 10);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// generic-proxy shared-memory writes -> visible to the tensor core / bulk copies
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// generic <-> async proxy ordering for global memory (a bulk copy's writes
// published through a flag, or a bulk copy reading what a flag published)
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void store_release_gpu(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int load_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_saddr, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// 32 consecutive fp32 columns of this thread's lane (no wait; see tmem_wait_ld)
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar`.  Gives up after `budget` clock cycles (or
// at once when *abort is already set): then sets *abort and returns false, so
// that every later wait of the kernel returns at once and the kernel runs to
// its end with the same control flow in every thread.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          long long budget = 4000000000LL) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (*abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > budget) {
      *abort = 1;
      return false;
    }
  }
}

// bulk copy global -> shared, completing `bytes` transactions on `bar`
__device__ __forceinline__ void bulk_g2s(uint32_t dst_saddr, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_saddr),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// bulk copy shared -> global, in the issuing thread's bulk async-group
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src_saddr, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(src_saddr), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the issuing thread's bulk stores have read their shared-memory sources
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// the same for all but the issuing thread's most recent bulk group
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// the issuing thread's bulk stores have completed
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// TMA: 3-D tiled load of box {x, y, z} at coordinates (x, y, z) of `tmap`
// (a __grid_constant__ CUtensorMap), completing transactions on `bar`
__device__ __forceinline__ void tma_load_3d(uint32_t dst_saddr, const void *tmap, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst_saddr),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Ampere-style asynchronous copies (4 or 16 bytes; src_bytes = 0 fills zeros)
__device__ __forceinline__ void cp_async4(uint32_t dst_saddr, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst_saddr), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst_saddr, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_saddr), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// wait for all of this thread's cp.async copies
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// arrive on `bar` once this thread's earlier cp.async copies have landed
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// named barrier among `nthreads` threads (a multiple of 32)
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace sm100
}  // namespace gdn
