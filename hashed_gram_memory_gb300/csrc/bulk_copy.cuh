// bulk_copy.cuh -- the inline-PTX pieces of the bulk-copy kernels (sm_103a):
// mbarrier set-up, arrival and polling, 1-D cp.async.bulk global -> shared
// copies completing on an mbarrier, L2 prefetch, a wait bounded by the global
// timer, and the host helper that raises a kernel's dynamic shared-memory
// ceiling once per device.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace engram {
namespace {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Asks L2 to fetch `bytes` (a multiple of 16) at `src` (16-byte aligned) ahead of use.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Polls the phase of `bar` with parity `parity` until it completes (true) or
// limit_ns passes (false).
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, int64_t limit_ns, uint32_t parity = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((int64_t)(global_ns() - t0) > limit_ns) return false;
  }
}

// Raises a kernel's dynamic shared-memory ceiling, once per device, to the 227 KB
// a block may use less the kernel's static shared memory (any launch's request
// fits under it).  `configured` is the kernel's own bit set of devices done.
template <typename Kernel>
cudaError_t raise_smem_ceiling(Kernel kern, std::atomic<uint64_t> &configured) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(227 * 1024 - fa.sharedSizeBytes));
  if (e == cudaSuccess) configured.fetch_or(bit, std::memory_order_release);
  return e;
}

}  // namespace
}  // namespace engram
