// Device-side helpers shared by the ig3 kernels: the bounded-wait machinery,
// the per-device status word, mbarrier / bulk-copy / tcgen05 wrappers written as
// inline PTX for sm_103a, and the fused activation.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ig3 {

// Bits of the per-device status word (a __device__ variable in ig3_api.cu whose
// address the host passes to every kernel that can wait).
enum : unsigned { kDevStatusTimeout = 1u };

// Everything a kernel needs to bound its waits.
struct WaitCtl {
  unsigned long long limit_ns;  // longest single wait before giving up
  unsigned int* status;         // device status word (atomicOr'ed on timeout)
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait until the barrier's phase with the given parity has completed, for at most
// ctl.limit_ns.  `abort` is a shared-memory flag the whole CTA watches: once any
// thread gives up, every other wait in the CTA returns false promptly too.  On a
// timeout the device status word records it.  Returns true if the phase completed.
static __device__ __noinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                               volatile int* abort) {
  const uint32_t addr = smem_addr(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > ctl.limit_ns) {
        *abort = 1;
        atomicOr(ctl.status, kDevStatusTimeout);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ bulk copies (TMA, 1-D)
// Global -> this CTA's shared memory, completion counted in bytes on `bar`.
// src, dst and bytes must all be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async proxy
// (tensor-core operand reads, bulk copies).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ activation
// tanh(mish(y)), mish(y) = y * tanh(softplus(y)).  With n = e^y,
// tanh(log(1 + n)) = ((1+n)^2 - 1) / ((1+n)^2 + 1) = n(n+2) / (n(n+2) + 2),
// so one exponential replaces exp + log1p + tanh.  For y > 15, tanh(softplus(y))
// differs from 1 by about 2e-13, below float resolution, so mish(y) = y.
__device__ __forceinline__ float tanh_mish(float y) {
  if (y > 15.0f) return tanhf(y);
  const float n = expf(y);
  const float t = n * (n + 2.0f);
  return tanhf(y * __fdividef(t, t + 2.0f));
}

}  // namespace ig3
