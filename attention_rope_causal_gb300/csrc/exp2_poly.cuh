// 2^x on the FMA pipes, for offloading part of the softmax exponentials from the MUFU unit.
//
// Method: Cody-Waite style range reduction (W. J. Cody and W. Waite, "Software Manual for the
// Elementary Functions", 1980): x = j + f with j = floor(x) and f in [0, 1); 2^f by a degree-3
// polynomial; 2^j applied by adding j to the exponent field.  The polynomial is a minimax fit of
// 2^f on [0, 1) in relative error made for this library (csrc/fit_exp2_poly.py, linear programming
// on a dense grid); realised fp32 error <= 7.5e-5 relative, below half an ulp of the fp16 P it feeds
// (4.9e-4) and far below bf16's.
//
// floor(x) comes from one round-toward-minus-infinity add of 1.5 * 2^23: in [2^23, 2^24) floats are
// spaced by 1, so the sum is exactly 1.5 * 2^23 + floor(x) and its bit pattern is that of 1.5 * 2^23
// plus floor(x); shifted left by 23 the constant part leaves the 32-bit word and floor(x) lands in the
// exponent field.  Inputs are clamped to >= -126 so the exponent never underflows past zero (the
// result there is < 2^-125, i.e. zero for a probability); softmax inputs never exceed +8.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace attnfuse {

constexpr float kExp2C0 = 0.9999251961708069f;
constexpr float kExp2C1 = 0.6958335638046265f;
constexpr float kExp2C2 = 0.22606714069843292f;
constexpr float kExp2C3 = 0.07802452892065048f;
constexpr float kExp2Magic = 12582912.0f;  // 1.5 * 2^23

// 2^x0, 2^x1 for the packed pair x = (x0, x1).
__device__ __forceinline__ void exp2_poly_pair(uint64_t x, float& p0, float& p1) {
  float x0, x1;
  ptx::f2_unpack(x, x0, x1);
  const uint64_t xc = ptx::f2_pack(fmaxf(x0, -126.f), fmaxf(x1, -126.f));
  const uint64_t magic = ptx::f2_pack(kExp2Magic, kExp2Magic);
  const uint64_t t = ptx::f2_add_rm(xc, magic);           // 1.5 * 2^23 + floor(x)
  const uint64_t f = ptx::f2_sub(xc, ptx::f2_sub(t, magic));  // x - floor(x), exact
  uint64_t q = ptx::f2_fma(ptx::f2_pack(kExp2C3, kExp2C3), f, ptx::f2_pack(kExp2C2, kExp2C2));
  q = ptx::f2_fma(q, f, ptx::f2_pack(kExp2C1, kExp2C1));
  q = ptx::f2_fma(q, f, ptx::f2_pack(kExp2C0, kExp2C0));
  float q0, q1, t0, t1;
  ptx::f2_unpack(q, q0, q1);
  ptx::f2_unpack(t, t0, t1);
  p0 = __uint_as_float(__float_as_uint(q0) + (__float_as_uint(t0) << 23));
  p1 = __uint_as_float(__float_as_uint(q1) + (__float_as_uint(t1) << 23));
}

}  // namespace attnfuse
