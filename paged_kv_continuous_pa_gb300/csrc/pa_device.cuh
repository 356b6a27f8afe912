// pa_device.cuh -- device-side building blocks shared by the paged-attention
// kernels: mbarriers, 1-D bulk (TMA engine) copies, element conversions and the
// status word.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pa_kernels.h"

namespace pa {

// ------------------------------------------------------------ status word --

// Record the first device-side error: compare-and-swap from PA_OK, so a
// later error never overwrites an earlier one.  Never traps.
__device__ __forceinline__ void record_error(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (the bulk-copy engine).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One poll of the phase with the given parity.  If the phase is not complete
// the thread may sleep in the poll for up to kWaitHintNs (the hardware wakes
// it when the phase completes), so waiting warps do not spin on the issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  if (kWaitHintNs > 0) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kWaitHintNs)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
  }
  return ok != 0;
}

// One poll of the phase with the given parity that never sleeps.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// if it has not completed after limit_us microseconds.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit_us) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  const uint64_t limit_ns = static_cast<uint64_t>(limit_us) * 1000u;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------- 1-D bulk copy (TMA) --

// Global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) by the bulk-copy engine; completion is counted on `bar` in bytes.
// The L2 policy marks the source evict-first: K/V pages are streamed once.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Barrier over the first NT threads of the CTA (named barrier 1), for code
// that runs in a CTA whose remaining warps have other work or have exited.
// A single warp (NT = 32) syncs on its own, so that code written for a
// one-warp CTA also runs in each warp of a wider one.
template <int NT>
__device__ __forceinline__ void sync_threads_n() {
  if constexpr (NT == 32)
    __syncwarp();
  else
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// Programmatic dependent launch.  A kernel launched as a dependent of the
// previous kernel in the stream may start before that kernel finishes;
// griddep_wait() returns once it has completed and its writes are visible
// (at once when the kernel was launched normally).  griddep_launch_dependents()
// lets the next kernel start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory accesses before its later
// async-proxy (bulk-copy) operations on shared memory.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Generic-proxy global memory accesses (another CTA's stores, ordered before
// this point by an acquire) before this thread's bulk copies read them.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// 2^x with the hardware approximation (ex2.approx.ftz.f32: relative error
// about 2^-22, subnormal results flushed to zero).  Softmax weights below
// 2^-126 contribute nothing at FP32 precision.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------ conversions --

// Two bf16 packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The K/V append's encoders (one definition for the append kernel and the
// attention units that append their own rows): fp32 -> bf16 round to nearest
// even; fp32 -> e4m3 as satfinite round-to-nearest-even of x / scale with one
// IEEE binary32 division.
__device__ __forceinline__ uint32_t encode_bf16(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

__device__ __forceinline__ uint32_t encode_e4m3(float x, float scale) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x, scale), __NV_SATFINITE, __NV_E4M3)) & 0xffu;
}

// Two e4m3 codes in the low 16 bits -> two floats, exactly (every e4m3 value is
// an f16 value), through the hardware e4m3x2 -> f16x2 conversion.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes & 0xffffu), __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

}  // namespace pa
