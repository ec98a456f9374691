// Shared pieces of the multi-query attention kernel on the 5th-generation
// tensor cores (tcgen05; the kernel itself is in pkv_prefill_tc05x2.cuh):
// tile size, the slack of the lazily raised exponent base, and the softmax
// helpers.
#pragma once

#include "pkv_prefill.cuh"
#include "pkv_umma.cuh"

namespace pkv {

// 2^x on the multi-function unit (flush-to-zero; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (a, b) -> bf16 pairs hi, lo with a ~ hi + lo, without conversion
// instructions: hi truncates a to its upper 16 bits, the remainder a - hi is
// exact in fp32 and is truncated the same way, so that 0 <= a - (hi + lo)
// < 2^-14 a for the finite non-negative a the softmax produces.  The two
// remainders are formed with one packed fp32x2 FMA.
__device__ __forceinline__ void split_bf16x2_trunc(float a, float b, uint32_t& hi, uint32_t& lo) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  const float2 t = make_float2(__uint_as_float(ua & 0xffff0000u), __uint_as_float(ub & 0xffff0000u));
  const float2 r = __ffma2_rn(t, make_float2(-1.f, -1.f), make_float2(a, b));
  hi = __byte_perm(ua, ub, 0x7632);
  lo = __byte_perm(__float_as_uint(r.x), __float_as_uint(r.y), 0x7632);
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

constexpr int kT5Rows = 128;     // query rows per tile: one M = 128 MMA
constexpr float kT5Slack = 8.f;  // raise the exponent base only past this (log2 units)

}  // namespace pkv
