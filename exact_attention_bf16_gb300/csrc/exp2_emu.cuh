// exp2 on the FMA/ALU pipes: Cody-Waite range split plus a cubic (wittx
// "FlashAttention-4", section 用软件"伪造"硬件指令; jsqmd "GPU 算力翻倍…
// FlashAttention-4", section 四.1):
//   2^x = 2^n * 2^f,  n = floor(x),  f = x - n in [0, 1),
//   2^f ~ p(f) = c0 + f (c1 + f (c2 + f c3))  (Horner, three FMAs),
//   2^n is added straight into p's IEEE-754 exponent field.
// The coefficients (exp2_poly_coeffs.h) are the minimax relative-error cubic
// with p(0) = 1 (so x = integer is exact), max relative error 8.6e-5.
// floor(x) is taken with a round-down add of 1.5 * 2^23, which leaves n in the
// low mantissa bits of the sum: no conversion instruction, so nothing runs on
// the special-function pipe. Inputs are clamped to >= -127; -inf gives +0.
#pragma once
#include "exp2_poly_coeffs.h"

namespace gb300 {

__device__ __forceinline__ float ex2_emu(float x) {
  constexpr float kShift = 12582912.0f;     // 1.5 * 2^23
  x = fmaxf(x, -127.0f);
  const float t = __fadd_rd(x, kShift);     // kShift + floor(x), exactly
  const float n = t - kShift;               // floor(x)
  const float f = x - n;                    // [0, 1)
  float p = fmaf(EXP2_POLY_C3, f, EXP2_POLY_C2);
  p = fmaf(p, f, EXP2_POLY_C1);
  p = fmaf(p, f, EXP2_POLY_C0);
  // low 9 bits of t's mantissa hold n (mod 512); shift them onto the exponent field
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

}  // namespace gb300
