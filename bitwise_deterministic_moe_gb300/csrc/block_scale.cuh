// Division by an NVFP4 block scale without a division instruction per element.
//
// The NVFP4 element code is E2M1(RN(a / s)) with a = RN(x * S_enc) and s the
// block's E4M3 scale value, so every element needs the correctly rounded
// binary32 quotient.  All sixteen elements of a block share s, so the block
// computes y = RN(1/s) once and each element takes Markstein's correction
// step (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Develop. 34(1), 1990):
//   q = RN(a * y)         within one ulp of a / s, since y is within half an ulp of 1/s
//   r = RN(a - s * q)     exact: the residual of a quotient within one ulp is representable
//   c = RN(q + r * y)     the correctly rounded quotient RN(a / s)
// provided nothing underflows.  For the scales an E4M3 code can hold
// (2^-9 <= s <= 448) and the elements an NVFP4 block can hold (|a / s| <= 6
// up to the scale's rounding), every quotient of magnitude >= 2^-3 is reached
// through normal numbers only; smaller quotients encode to a signed zero
// whatever their last bits.  One rounding of the fma can turn the zero
// quotient -0 into +0 (-0 + +0 = +0), so the sign of a is copied onto the
// result, which is exact for every other quotient (its sign is already a's).
// The GPU tests compare this routine with the compiler's correctly rounded
// division on every binary32 significand for every E4M3 scale value.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace dmoe {

// two quotients at a time on the packed fp32x2 pipe; nb = (-s, -s), y = (RN(1/s), RN(1/s))
__device__ __forceinline__ float2 div2_by_block_scale(float2 a, float2 nb, float2 y) {
  const float2 q = __fmul2_rn(a, y);
  const float2 r = __ffma2_rn(q, nb, a);   // a - s q, exact
  const float2 c = __ffma2_rn(r, y, q);
  return make_float2(__uint_as_float(__float_as_uint(c.x) | (__float_as_uint(a.x) & 0x80000000u)),
                     __uint_as_float(__float_as_uint(c.y) | (__float_as_uint(a.y) & 0x80000000u)));
}

}  // namespace dmoe
