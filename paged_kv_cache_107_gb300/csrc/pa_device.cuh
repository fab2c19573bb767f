// pa_device.cuh — device-side building blocks shared by the library's kernels:
// mbarrier and bulk-copy PTX wrappers, bounded waits, bf16 unpacking, error flags.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

constexpr int kHeadDim = 128;
// SM clock cycles before a wait is declared stuck (about 0.13 s at 2 GHz; a healthy wait in
// these pipelines lasts microseconds), so a broken pipeline ends instead of hanging. A test
// build of the library defines PA_WAIT_CYCLES smaller to make a wait run out on purpose.
#ifndef PA_WAIT_CYCLES
#define PA_WAIT_CYCLES (1ll << 28)
#endif
constexpr long long kWaitCycles = PA_WAIT_CYCLES;

__device__ __forceinline__ void set_dev_err(int* dev_err, int bit) {
  if (dev_err) atomicOr(dev_err, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Bounded wait on phase `parity`. Returns false (and leaves the barrier alone) if the
// phase did not complete within the limit; *abort makes later waits give up at once.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long limit = (abort && *abort) ? 4096ll : kWaitCycles;
  const long long t0 = clock64();
  while (clock64() - t0 < limit) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}

// Bounded wait for this CTA's own copies in flight (before it exits): the full limit even
// after another wait gave up, because a copy still landing in shared memory must not outlive
// the CTA; copies end in microseconds unless the memory system is broken.
__device__ __forceinline__ bool mbar_wait_copies(uint64_t* bar, uint32_t parity) {
  return mbar_wait(bar, parity, nullptr);
}

// ---------------------------------------------------------------- bulk copies
// One contiguous global -> shared copy, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (the K/V stream is read once).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Bulk prefetch of [src, src + bytes) into L2 (src 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- dependent launches
// With programmatic stream serialization the next grid may start while this one runs:
// launch_dependents lets it be scheduled; wait blocks until every grid this one depends
// on has completed and its memory operations are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- shared loads
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ float4 lds128f(const void* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// ---------------------------------------------------------------- bf16 <-> f32
// A 32-bit word holds two bf16 values, element 0 in the low half. A bf16 is the top 16
// bits of an fp32, so widening is a shift or a mask.
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  bf16x2_to_f32(v.x, f[0], f[1]);
  bf16x2_to_f32(v.y, f[2], f[3]);
  bf16x2_to_f32(v.z, f[4], f[5]);
  bf16x2_to_f32(v.w, f[6], f[7]);
}

// Round-to-nearest-even packing of two fp32 values into bf16x2 (hardware cvt).
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace pa
