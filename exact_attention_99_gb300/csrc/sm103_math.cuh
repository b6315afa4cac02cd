// Packed fp32 arithmetic (f32x2) and the software exp2 used by the softmax
// warps, for sm_103a.
#pragma once
#include <cstdint>

#include "exp2_poly.h"

namespace fa {

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x for a pair of arguments on the FMA pipes: round-to-nearest split
// x = n + f (adding 1.5*2^23 rounds to an integer and leaves n in the low
// mantissa bits), degree-3 minimax polynomial for 2^f on [-1/2, 1/2], times
// 2^n built directly from its exponent bits. Arguments are clamped to -127,
// where 2^n has exponent field 0 and the result is exactly 0.
__device__ __forceinline__ void exp2_poly_pair(float& a, float& b) {
  a = fmaxf(a, -127.0f);
  b = fmaxf(b, -127.0f);
  const uint64_t magic = pack2(12582912.0f, 12582912.0f);
  const uint64_t x = pack2(a, b);
  const uint64_t t = fadd2(x, magic);
  const uint64_t n = fadd2(t, pack2(-12582912.0f, -12582912.0f));
  const uint64_t f = fadd2(x, n ^ 0x8000000080000000ull);  // x - n
  uint64_t q = ffma2(pack2(FA_EXP2_C3, FA_EXP2_C3), f, pack2(FA_EXP2_C2, FA_EXP2_C2));
  q = ffma2(q, f, pack2(FA_EXP2_C1, FA_EXP2_C1));
  q = ffma2(q, f, pack2(FA_EXP2_C0, FA_EXP2_C0));
  float ta, tb;
  unpack2(t, ta, tb);
  // low bits of t hold n; (n + 127) << 23 is the bit pattern of 2^n (0 for n = -127)
  const uint64_t sc = pack2(__int_as_float((__float_as_int(ta) + 127) << 23),
                            __int_as_float((__float_as_int(tb) + 127) << 23));
  unpack2(fmul2(q, sc), a, b);
}

}  // namespace fa
