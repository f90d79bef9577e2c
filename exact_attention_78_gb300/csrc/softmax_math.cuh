// Exponential paths of the softmax, shared by the attention kernels and the
// exp2 self-check kernel so that the check exercises the very same code.
#pragma once

#include "exp2_poly.h"
#include "ptx.cuh"

namespace fa {

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

// Column `col` of a row uses the polynomial when (col mod 16) < EMU, the
// hardware exponential otherwise: EMU of every 16 entries go to the FMA pipe.
template <int EMU>
FA_DEV float exp2_mixed(float x, int col) {
  if (EMU > 0 && (col & 15) < EMU) return exp2_fma(x);
  return ex2_mufu(x);
}

}  // namespace fa
