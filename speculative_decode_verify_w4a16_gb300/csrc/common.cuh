// Shared device helpers for the w4a16sv kernels: mbarriers with bounded
// waits, 1-D bulk async copies (TMA engine), fences and the device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

// Bits of the device error word.
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrInput = 2u;
constexpr unsigned kErrBounds = 4u;  // bounds-checked builds: a computed index left its buffer

// Upper bound on any spin wait inside a kernel (ns of %globaltimer). A
// debug build of the library (for the tests that make a wait run out) sets
// a few milliseconds instead.
#ifndef W4A16_WAIT_LIMIT_NS
#define W4A16_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr unsigned long long kWaitLimitNs = W4A16_WAIT_LIMIT_NS;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// Bounds-checked builds (-DW4A16_BOUNDS_CHECK=1, a separate debug library)
// test every instrumented global index against its buffer: one outside
// [0, limit) sets kErrBounds in the device error word and the access is
// skipped (no trap). In the product build this is always true and costs
// nothing.
#ifndef W4A16_BOUNDS_CHECK
#define W4A16_BOUNDS_CHECK 0
#endif
__device__ __forceinline__ bool in_bounds(unsigned* err, int64_t idx, int64_t limit) {
#if W4A16_BOUNDS_CHECK
  if (idx < 0 || idx >= limit) {
    report_error(err, kErrBounds);
    return false;
  }
#else
  (void)err;
  (void)idx;
  (void)limit;
#endif
  return true;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Test for completion of the phase with the given parity; if it is not
// complete the thread may sleep in hardware for up to `hint_ns` before the
// test returns false (so waiting warps do not spin through issue slots).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns = 0) {
  uint32_t ok;
  if (hint_ns == 0) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
  }
  return ok != 0;
}

// Non-blocking test for completion of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, sleeping in hardware
// between tests. Gives up after kWaitLimitNs, records kErrTimeout and returns
// false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err) {
  if (mbar_try_wait(bar, parity, 1000000u)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity, 1000000u)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report_error(err, kErrTimeout);
      return false;
    }
  }
}

// ------------------------------------------------------- bulk async copies
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes).
// src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority policy (streamed-once data).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------- programmatic dependent launch
// Kernels are launched with programmatic stream serialisation: they may start
// while the previous kernel on the stream is still running. Everything that
// reads or writes global memory shared with other kernels (inputs, outputs,
// workspace) comes after grid_dependency_wait(), which returns once the
// preceding grid has completed and its writes are visible. Without the launch
// attribute both instructions are no-ops.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------- atomics
// Device-scope fetch-add with acquire-release semantics: publishes this
// thread's earlier writes (and those ordered before them, e.g. by __syncwarp)
// and makes writes published by earlier adders visible to later reads.
__device__ __forceinline__ int atomic_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Device-scope acquire load: reading the value the last of a series of
// atom.acq_rel adds wrote makes every adder's earlier writes visible to this
// thread's later reads.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// --------------------------------------------------------- packed fp32 math
// (d0, d1) = (a0 * b0 + d0, a1 * b1 + d1): two IEEE fp32 fused multiply-adds
// (round to nearest each, the same results as two fmaf) in one instruction.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rd, {%0, %1};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rd;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// exp(a - b) for finite fp32 a <= b, for values that decide a draw or an
// acceptance: the difference is formed exactly as hi + lo (TwoSum, Knuth,
// TAOCP vol. 2, 4.2.2; |lo| <= 2^-24 |hi|) and exp(hi + lo) = exp(hi) (1 + lo)
// to within lo^2 / 2; exp(hi) is the library's accurate expf (the fast
// approximation's error grows with |hi|).
__device__ __forceinline__ float exp_of_diff(float a, float b) {
  const float s = __fsub_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float lo = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(-b, bb));
  const float e = expf(s);
  return __fmaf_rn(e, lo, e);
}

// ------------------------------------------------------------ shared loads
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// -------------------------------------------------------- global loads
__device__ __forceinline__ float4 ldg_stream_f4(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// the same with an L2 eviction-priority policy (createpolicy)
__device__ __forceinline__ float4 ldg_hint_f4(const float4* p, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ float ldg_stream_f(const float* p) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

}  // namespace w4a16
