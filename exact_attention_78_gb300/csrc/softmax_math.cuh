// Exponential paths of the softmax, shared by the attention kernels and the
// exp2 self-check kernel so that the check exercises the very same code.
#pragma once

#include "exp2_poly.h"
#include "ptx.cuh"

namespace fa {

// ------------------------------------------------ packed FP32 pairs (sm_100+) --
// Two floats in one 64-bit register pair; the .f32x2 forms of add/mul/fma
// process both in one instruction.

FA_DEV uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
FA_DEV void up2(uint64_t v, float& lo, float& hi) { asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v)); }
FA_DEV uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
FA_DEV uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
FA_DEV uint64_t add2_rm(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rm.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
FA_DEV uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three floats in one instruction
FA_DEV float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x on the FMA pipe ("FlashAttention-4: Algorithm and Kernel Pipelining
// Co-Design for Asymmetric Hardware Scaling", fdeinterviews.com summary, bullet
// "Software exponentials"): x = n + f with n = floor(x) and f in [0, 1);
// p(f) ~ 2^f by Horner's rule; n is added to the exponent field of p(f).
// The floor comes from adding 1.5 * 2^23 with rounding toward minus
// infinity, which leaves n in the low mantissa bits of the sum.  x is clamped
// at -127 first (masked entries arrive as -inf and come out as exactly 0;
// anything that small is negligible next to a row sum of at least 1).
FA_DEV float exp2_fma(float x) {
  x = fmaxf(x, -127.0f);
  const float big = __fadd_rd(x, 12582912.0f);  // 1.5 * 2^23 + floor(x)
  const float n = big - 12582912.0f;            // exact
  const float f = x - n;                        // exact, in [0, 1)
  float p = fmaf(FA_EXP2_C3, f, FA_EXP2_C2);
  p = fmaf(p, f, FA_EXP2_C1);
  p = fmaf(p, f, FA_EXP2_C0);
  // bits(big) << 23 equals n << 23 modulo 2^32: the constant part
  // 0x4B400000 has nine zero bits at positions 0..8
  return __uint_as_float(__float_as_uint(p) + (__float_as_uint(big) << 23));
}

// The same polynomial for two arguments with packed FP32x2 instructions.
FA_DEV void exp2_fma2(float x0, float x1, float& y0, float& y1) {
  const uint64_t x = pk2(fmaxf(x0, -127.0f), fmaxf(x1, -127.0f));
  const uint64_t big = add2_rm(x, pk2(12582912.0f, 12582912.0f));   // 1.5 * 2^23 + floor(x)
  const uint64_t n = add2(big, pk2(-12582912.0f, -12582912.0f));    // exact
  const uint64_t f = fma2(n, pk2(-1.0f, -1.0f), x);                  // x - n, exact
  uint64_t p = fma2(pk2(FA_EXP2_C3, FA_EXP2_C3), f, pk2(FA_EXP2_C2, FA_EXP2_C2));
  p = fma2(p, f, pk2(FA_EXP2_C1, FA_EXP2_C1));
  p = fma2(p, f, pk2(FA_EXP2_C0, FA_EXP2_C0));
  float p0, p1, b0, b1;
  up2(p, p0, p1);
  up2(big, b0, b1);
  y0 = __uint_as_float(__float_as_uint(p0) + (__float_as_uint(b0) << 23));
  y1 = __uint_as_float(__float_as_uint(p1) + (__float_as_uint(b1) << 23));
}

// Columns c, c+1 (c even) of a row: the pair uses the polynomial when
// (c mod 16) < EMU, the hardware exponential otherwise, so EMU of every 16
// entries go to the FMA pipe.
template <int EMU>
FA_DEV void exp2_pair(float x0, float x1, int c, float& y0, float& y1) {
  if (EMU > 0 && (c & 15) < EMU) {
    exp2_fma2(x0, x1, y0, y1);
  } else {
    y0 = ex2_mufu(x0);
    y1 = ex2_mufu(x1);
  }
}

}  // namespace fa
