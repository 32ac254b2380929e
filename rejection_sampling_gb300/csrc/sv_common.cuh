// sv_common.cuh -- device helpers shared by the verification kernels (sm_103a).
//
// Inline PTX for the pieces CUDA C++ does not expose directly: mbarrier
// init/arrive/expect-tx/try-wait, the 1-D bulk copy global -> shared
// (cp.async.bulk, completed through an mbarrier transaction count), and the
// ex2.approx instruction.  No CUDA math-library internals are reproduced.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sv_internal.h"

namespace sv {

// log2(e) rounded to fp32: exp(v - m) = 2^((v - m) * log2 e).  Every kernel
// and every combination step uses this one constant, so the scale of the
// partial sums and of the gathered probabilities agree exactly.
constexpr float kLog2e = 1.44269504088896340736f;

// ---------------------------------------------------------------------------
// fast exp2 (MUFU.EX2): ex2.approx.ftz.f32, hardware instruction
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 pair in one 32-bit word -> two exact fp32 values
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// max of two bf16 pairs (exact; NaN operands are ignored like IEEE maxNum)
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---------------------------------------------------------------------------
// packed fp32 pairs (sm_100+ f32x2 arithmetic: two IEEE fp32 operations per
// instruction, each rounded exactly as its scalar form)
// ---------------------------------------------------------------------------
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(f32x2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// ---------------------------------------------------------------------------
// warp reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// exclusive prefix over lanes (fp64)
__device__ __forceinline__ double warp_exclusive_scan_d(double v, int lane) {
  double x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x - v;
}

// ---------------------------------------------------------------------------
// mbarrier (shared memory, CTA scope)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with `parity` (never suspends the warp; for
// polling loops in which the lanes of a warp watch different barriers).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase with `parity` completed, false if the
// bound (in SM clock cycles) ran out first.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long bound_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > bound_cycles) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// 1-D bulk copy global -> shared::cta, completion on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// global-memory flags with acquire / release semantics (GPU scope)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// acquire-release fence at GPU scope: orders this thread's earlier memory
// operations before its later ones for every observer on the GPU (lighter than
// the sequentially consistent fence of __threadfence)
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void nanosleep_ns(uint32_t ns) {
  asm volatile("nanosleep.u32 %0;" ::"r"(ns));
}

}  // namespace sv

namespace sv {

// ---------------------------------------------------------------------------
// float-float arithmetic (a value is hi + lo with |lo| <= ulp(hi)/2).
// GB300's fp64 pipe is a small fraction of its fp32 rate, so sums that need
// more than fp32 precision are carried as unevaluated pairs of floats, using
// the error-free transformations two-sum (Knuth) and two-product (FMA).
// Explicit _rn intrinsics keep the compiler from contracting or reordering.
// ---------------------------------------------------------------------------
struct ff {
  float hi, lo;
};

__device__ __forceinline__ ff ff_make(float a) { return ff{a, 0.f}; }

// s + e == a + b exactly
__device__ __forceinline__ ff two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bv = __fsub_rn(s, a);
  const float av = __fsub_rn(s, bv);
  const float e = __fadd_rn(__fsub_rn(a, av), __fsub_rn(b, bv));
  return ff{s, e};
}

// renormalise (|b| <= |a| or a == 0)
__device__ __forceinline__ ff quick_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return ff{s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
  ff s = two_sum(a.hi, b.hi);
  const float e = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
  return quick_two_sum(s.hi, e);
}

__device__ __forceinline__ ff ff_add_f(ff a, float b) {
  ff s = two_sum(a.hi, b);
  return quick_two_sum(s.hi, __fadd_rn(s.lo, a.lo));
}

__device__ __forceinline__ ff ff_neg(ff a) { return ff{-a.hi, -a.lo}; }
__device__ __forceinline__ ff ff_sub(ff a, ff b) { return ff_add(a, ff_neg(b)); }

// a * b for floats, exactly as a pair
__device__ __forceinline__ ff two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return ff{p, __fmaf_rn(a, b, -p)};
}

// ff * float
__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
  ff p = two_prod(a.hi, b);
  return quick_two_sum(p.hi, __fmaf_rn(a.lo, b, p.lo));
}

__device__ __forceinline__ float ff_to_f(ff a) { return __fadd_rn(a.hi, a.lo); }

// sign of a - b
__device__ __forceinline__ bool ff_gt(ff a, ff b) {
  const ff d = ff_sub(a, b);
  return d.hi > 0.f || (d.hi == 0.f && d.lo > 0.f);
}

__device__ __forceinline__ ff ff_shfl(ff a, int src) {
  return ff{__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}
__device__ __forceinline__ ff ff_shfl_up(ff a, int d) {
  return ff{__shfl_up_sync(0xffffffffu, a.hi, d), __shfl_up_sync(0xffffffffu, a.lo, d)};
}
__device__ __forceinline__ ff ff_shfl_xor(ff a, int m) {
  return ff{__shfl_xor_sync(0xffffffffu, a.hi, m), __shfl_xor_sync(0xffffffffu, a.lo, m)};
}

__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
  return v;
}

// exclusive prefix over lanes
__device__ __forceinline__ ff warp_exclusive_scan_ff(ff v, int lane) {
  ff x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff y = ff_shfl_up(x, o);
    if (lane >= o) x = ff_add(x, y);
  }
  return ff_sub(x, v);
}

}  // namespace sv
