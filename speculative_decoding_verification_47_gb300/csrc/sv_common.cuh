// Device helpers shared by the verify, commit and LM-head kernels (sm_103a).
//
// Bulk asynchronous copies (the TMA engine's 1-D form), mbarrier completion,
// thread-block-cluster distributed shared memory, and double-float ("two
// float") accumulation.  The double-float sum keeps a row's normaliser and the
// residual CDF accurate to ~1e-9 relative, which the verify step needs so that
// its token decisions agree with exact arithmetic except when the exact
// decision itself sits within ~1e-9 of its threshold.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cooperative_groups.h>

namespace sv {

namespace cg = cooperative_groups;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarriers (the LM head's TMA copies complete on them)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// try_wait that may suspend the thread for up to `hint_ns` before returning.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait by ONE thread (the others sleep at the following CTA barrier
// instead of spinning): each try suspends for up to 0.5 ms; after `limit`
// failed tries (about a second) the caller gets false and reports a timeout
// instead of waiting forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t limit = 2048) {
  for (uint32_t it = 0; it < limit; ++it)
    if (mbar_try_wait_hint(bar, parity, 500000u)) return true;
  return false;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor in the stream still runs;
// pdl_wait() blocks until that predecessor has completed and its memory
// operations are visible (it returns at once when there is none).
// pdl_launch_dependents() lets the next such kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Exponential: 2^x on the MUFU unit (flush-to-zero below 2^-126).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Double-float accumulation (Knuth's two-sum; no reassociation: this file is
// compiled without fast-math).
// ---------------------------------------------------------------------------
struct DF {
  float hi, lo;
};

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// acc += x, keeping the rounding error in acc.lo (renormalised lazily).
__device__ __forceinline__ void df_acc(DF& acc, float x) {
  float s, e;
  two_sum(acc.hi, x, s, e);
  acc.hi = s;
  acc.lo = __fadd_rn(acc.lo, e);
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  float hi = __fadd_rn(s, e);
  return DF{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}

__device__ __forceinline__ DF df_shfl_xor(DF v, int mask) {
  return DF{__shfl_xor_sync(0xffffffffu, v.hi, mask), __shfl_xor_sync(0xffffffffu, v.lo, mask)};
}

__device__ __forceinline__ DF df_warp_sum(DF v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = df_add(v, df_shfl_xor(v, m));
  return v;
}

__device__ __forceinline__ DF df_neg(DF a) { return DF{-a.hi, -a.lo}; }

__device__ __forceinline__ DF df_sub(DF a, DF b) { return df_add(a, df_neg(b)); }

// sign of a - b (double-float compare without FP64 instructions)
__device__ __forceinline__ bool df_gt(DF a, DF b) {
  DF d = df_sub(a, b);
  return d.hi > 0.f || (d.hi == 0.f && d.lo > 0.f);
}

__device__ __forceinline__ bool df_pos(DF a) { return a.hi > 0.f || (a.hi == 0.f && a.lo > 0.f); }

// a * x for a float x (Dekker product with FMA)
__device__ __forceinline__ DF df_mul_f(DF a, float x) {
  float p = __fmul_rn(a.hi, x);
  float e = __fmaf_rn(a.hi, x, -p);
  e = __fmaf_rn(a.lo, x, e);
  float hi = __fadd_rn(p, e);
  return DF{hi, __fsub_rn(e, __fsub_rn(hi, p))};
}

// a / b in double-float: quotient, exact remainder, corrected quotient (the
// double-length division of T. J. Dekker, "A floating-point technique for
// extending the available precision", 1971), with float instructions only
__device__ __forceinline__ DF df_div(DF a, DF b) {
  float q1 = __fdiv_rn(a.hi, b.hi);
  DF r = df_sub(a, df_mul_f(b, q1));
  float q2 = __fdiv_rn(r.hi, b.hi);
  float hi = __fadd_rn(q1, q2);
  return DF{hi, __fsub_rn(q2, __fsub_rn(hi, q1))};
}

__device__ __forceinline__ float df_to_float(DF v) { return __fadd_rn(v.hi, v.lo); }

// ---------------------------------------------------------------------------
// Packed fp32 pairs (Blackwell f32x2 FMA / ADD: two lanes per instruction,
// each lane rounded exactly like its scalar counterpart).
// ---------------------------------------------------------------------------
typedef unsigned long long F2;

__device__ __forceinline__ F2 f2_pack(float a, float b) {
  F2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(F2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
  F2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  F2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// ---------------------------------------------------------------------------
// bf16 unpacking: word w holds element 2k in its low half, 2k+1 in its high.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace sv
