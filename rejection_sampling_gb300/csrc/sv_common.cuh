// sv_common.cuh -- device helpers shared by the verification kernels (sm_103a).
//
// Inline PTX for the pieces CUDA C++ does not expose directly (the
// ex2.approx instruction, bf16 pair maxima), warp reductions and scans, and
// float-float (pairs of fp32) arithmetic.  No CUDA math-library internals
// are reproduced.
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
// fast exp2 (MUFU.EX2): ex2.approx.ftz.f32, hardware instruction.  ex2 may be
// scheduled freely; ex2_ordered stays in program order with the other
// volatile asm (copy issue, waits), which the dense statistics stream
// measured faster with (its loads stay ahead of the arithmetic), while the
// warp-per-row and commit kernels measured faster with the free form.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ex2_ordered(float x) {
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
// packed fp32 pairs (add / fma .f32x2 on a 64-bit register pair): one issue
// slot for two round-to-nearest operations, each rounded exactly as the
// scalar instruction would round it
// ---------------------------------------------------------------------------
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2_pack(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(f32x2 r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// (2^(a0 L - c), 2^(a1 L - c)) for the pair (a0, a1): one packed fma, two ex2
__device__ __forceinline__ f32x2 f2_exp2_shift(f32x2 a, f32x2 L, f32x2 nc) {
  float y0, y1;
  f2_unpack(f2_fma(a, L, nc), y0, y1);
  return f2_pack(ex2(y0), ex2(y1));
}
__device__ __forceinline__ f32x2 f2_exp2_shift_ordered(f32x2 a, f32x2 L, f32x2 nc) {
  float y0, y1;
  f2_unpack(f2_fma(a, L, nc), y0, y1);
  return f2_pack(ex2_ordered(y0), ex2_ordered(y1));
}
// a bf16 pair in one 32-bit word as an fp32 pair (exact)
__device__ __forceinline__ f32x2 f2_bf16(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may be scheduled while its predecessor on the stream is still
// running; this waits until that grid has completed (and its memory is
// visible) before anything is read, then lets the next grid be scheduled
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
// ---------------------------------------------------------------------------
// shared-memory addresses for inline PTX
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarriers and bulk (TMA) copies into shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// make the initialised barriers visible to the async proxy (the bulk copies)
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// one test of the barrier's phase; a thread whose phase is not complete is
// suspended in hardware (up to kSuspendNs) rather than spinning on issue slots
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// wait for phase `parity` of a copy barrier until the globaltimer passes
// `deadline` (and for at most 2^28 polls)
static __device__ __noinline__ bool mbar_wait_until(uint64_t* bar, unsigned parity,
                                             unsigned long long deadline) {
  for (uint32_t i = 0; i < (1u << 28); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u && globaltimer() > deadline) return false;
  }
  return false;
}
// global -> this CTA's shared memory, completion counted on `bar`
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Row b's count of pieces whose statistics records are stored (the dense
// two-kernel path; one counter per 128-byte line).  A statistics warp adds
// its pieces of row b once the last of its records in that row is stored
// (release); the row kernel's thread 0 waits for the complete count before
// the row's records are read, and the row kernel clears it again.
__device__ __forceinline__ uint32_t* row_count(const DenseParams& P, int b) {
  return reinterpret_cast<uint32_t*>(P.ws + P.L.rcnt) + (size_t)b * kRowCountStride;
}
__device__ __forceinline__ void row_signal(const DenseParams& P, int b, long long pieces,
                                           int lane) {
  if (lane == 0)
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(row_count(P, b)),
                 "r"((uint32_t)pieces)
                 : "memory");
}
constexpr unsigned long long kRowWaitNs = 1000000000ull;  // one second
// Poll row b's count until it reaches `need`: relaxed loads 256 ns apart
// (an acquire load per poll costs the SM more), then one acquire load of the
// complete count.  At most a second of globaltimer and 2^22 polls; false when
// the wait ran out.
static __device__ __noinline__ bool wait_row_ready(const DenseParams& P, int b, uint32_t need) {
  const uint32_t* c = row_count(P, b);
  const unsigned long long deadline = globaltimer() + kRowWaitNs;
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    if (v >= need) {
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
      return true;
    }
    if (globaltimer() > deadline) return false;
    __nanosleep(256);
  }
  return false;
}

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

// ---------------------------------------------------------------------------
// partial softmax sums with integer reference points.  A partial sum is
// S = sum 2^(v log2e - c) with c = ceil(log2e * max v): every rescale between
// partials is then an exact power of two, formed on the integer pipe (no
// MUFU, no rounding).
// ---------------------------------------------------------------------------
// 2^d for an integer-valued d <= 0 (0 below the normal range, and for NaN)
__device__ __forceinline__ float pow2i(float d) {
  return d > -127.f ? __int_as_float(((int)d + 127) << 23) : 0.f;
}
// the reference point of a partial whose largest element is m
__device__ __forceinline__ float ref_point(float m) {
  return (m == -INFINITY) ? -INFINITY : ceilf(m * kLog2e);
}
// 2^(c - C): a partial with reference c moved to reference C >= c (0 for an
// all -inf partial)
__device__ __forceinline__ float scale_exact(float c, float C) {
  return (c == -INFINITY) ? 0.f : pow2i(c - C);
}
// order-preserving map of fp32 onto int32, so one redux.sync finds a warp's
// largest float
__device__ __forceinline__ int f2ord(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float ord2f(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7FFFFFFF); }

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

// warp-wide combination of per-lane (C, S) partials of two rows: the
// reference points by redux.sync, the exactly rescaled sums by one shuffle
// tree (float-float); every lane ends with the warp's totals
__device__ __forceinline__ void warp_combine_pair(float& Ct, ff& St, float& Cd, ff& Sd) {
  const float Cwt = ord2f(__reduce_max_sync(0xffffffffu, f2ord(Ct)));
  const float Cwd = ord2f(__reduce_max_sync(0xffffffffu, f2ord(Cd)));
  St = ff_mul_f(St, scale_exact(Ct, Cwt));
  Sd = ff_mul_f(Sd, scale_exact(Cd, Cwd));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const ff a = ff_shfl_xor(St, o), b = ff_shfl_xor(Sd, o);
    St = ff_add(St, a);
    Sd = ff_add(Sd, b);
  }
  Ct = Cwt;
  Cd = Cwd;
}

}  // namespace sv
