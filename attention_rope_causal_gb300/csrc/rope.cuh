// Rotary position embedding on the device: angles, cos/sin and the rotation of one 16-byte chunk
// pair.  Shared by the pre-rotation kernel and the fused attention kernel so that both rotate Q
// with bit-identical arithmetic.
//
// Convention (the pages name RoPE as a pre-multiplication transform of Q and K -- "AttnFuse Makes
// RoPE a First-Class Attention Compilation Operation", 2026-09-13 AI papers report, paragraph 1 --
// and print no formula; this library fixes the half-split form):
//   theta_k = base^(-2k/d),  pairs (k, k + d/2),  angle = p * theta_k with p the token index,
//   x'[k] = x[k] cos - x[k+d/2] sin,   x'[k+d/2] = x[k+d/2] cos + x[k] sin.
//
// Angles.  p * theta_k reaches 3.3e4 rad at p = 32767, where an fp32 product is off by up to
// ~2e-3 rad.  Instead the host stores, per pair k, the frequency in turns as a 64-bit fixed-point
// fraction F_k = round(theta_k / (2 pi) * 2^64).  The angle in turns, reduced modulo one turn, is
// then bits [32, 64) of the integer product p * F_k (two integer instructions).  That 32-bit turn
// fraction is reduced exactly, in integers, to the nearest quarter turn q and a remainder r in
// [-1/2, 1/2) quarter turns; sin and cos of (pi/2) r come from minimax polynomials (odd degree 7,
// even degree 8) fitted for this library (csrc/fit_sincos_poly.py; fp32 error <= 1.1e-7), and the
// quarter turns swap and negate them.  Angle error: 2^-32 turn from truncation plus one fp32
// rounding of r (< 5e-8 rad).  No table and no library call: the cost is fixed (~25 instructions).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace attnfuse {

constexpr int kMaxHalfDim = 64;  // d <= 128

struct RopeFreqs {
  uint32_t lo[kMaxHalfDim];  // low  32 bits of F_k
  uint32_t hi[kMaxHalfDim];  // high 32 bits of F_k
};

// cos and sin of 2 pi t / 2^32 for a 32-bit turn fraction t.
__device__ __forceinline__ void sincos_turns(uint32_t t, float& c, float& s) {
  const uint32_t q = (t + 0x20000000u) >> 30;                  // nearest quarter turn, mod 4
  const int32_t rem = (int32_t)(t - (q << 30));                // in [-2^29, 2^29)
  const float r = (float)rem * 9.313225746154785e-10f;         // * 2^-30: quarter turns in [-1/2, 1/2)
  const float z = __fmul_rn(r, r);
  const float sp = __fmul_rn(
      __fmaf_rn(__fmaf_rn(__fmaf_rn(-0.004624062217772007f, z, 0.07968810945749283f), z, -0.6459640860557556f), z,
                1.5707963705062866f),
      r);
  const float cp = __fmaf_rn(
      __fmaf_rn(__fmaf_rn(__fmaf_rn(0.0009058757568709552f, z, -0.020861255005002022f), z, 0.2536693811416626f), z,
                -1.2337005138397217f),
      z, 1.0f);
  // rotate (cp, sp) by q quarter turns
  const float c0 = (q & 1u) ? -sp : cp;
  const float s0 = (q & 1u) ? cp : sp;
  c = (q & 2u) ? -c0 : c0;
  s = (q & 2u) ? -s0 : s0;
}

// cos and sin of pos * theta_k, given F_k split into (flo, fhi).
__device__ __forceinline__ void rope_cs(uint32_t pos, uint32_t flo, uint32_t fhi, float& c, float& s) {
  const uint32_t turns = __umulhi(pos, flo) + pos * fhi;  // bits [32,64) of pos * F_k (mod 2^64)
  sincos_turns(turns, c, s);
}

// The same for any signed position: the turn fraction of -m is the negated turn fraction of m
// (within the 2^-32 turn truncation).
__device__ __forceinline__ void rope_cs_signed(int32_t pos, uint32_t flo, uint32_t fhi, float& c, float& s) {
  const uint32_t a = pos < 0 ? 0u - (uint32_t)pos : (uint32_t)pos;
  const uint32_t t = __umulhi(a, flo) + a * fhi;
  sincos_turns(pos < 0 ? 0u - t : t, c, s);
}

// (c, s) <- (c, s) * (c2, s2) as unit complex numbers: the angle advances by the angle of (c2, s2).
__device__ __forceinline__ void rope_advance(float& c, float& s, float c2, float s2) {
  float cn = __fmaf_rn(c, c2, -__fmul_rn(s, s2));
  float sn = __fmaf_rn(s, c2, __fmul_rn(c, s2));
  c = cn;
  s = sn;
}

// One rotated pair.  Written with explicit round-to-nearest intrinsics so no kernel can contract it
// differently: every caller gets bit-identical results for equal inputs.
__device__ __forceinline__ void rope_pair(float x, float y, float c, float s, float& xr, float& yr) {
  xr = __fmaf_rn(x, c, -__fmul_rn(y, s));
  yr = __fmaf_rn(y, c, __fmul_rn(x, s));
}

template <bool BF16>
struct Pack;

template <>
struct Pack<true> {
  __device__ __forceinline__ static void unpack(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};

template <>
struct Pack<false> {
  __device__ __forceinline__ static void unpack(uint32_t w, float& lo, float& hi) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};

// Rotate 8 pairs held as two 16-byte chunks: xv = elements [k0, k0+8), yv = [k0+d/2, k0+d/2+8).
template <bool BF16>
__device__ __forceinline__ void rope_rotate_chunk(uint4& xv, uint4& yv, const float (&c)[8], const float (&s)[8]) {
  uint32_t* xw = reinterpret_cast<uint32_t*>(&xv);
  uint32_t* yw = reinterpret_cast<uint32_t*>(&yv);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float x0, x1, y0, y1, a0, a1, b0, b1;
    Pack<BF16>::unpack(xw[w], x0, x1);
    Pack<BF16>::unpack(yw[w], y0, y1);
    rope_pair(x0, y0, c[2 * w], s[2 * w], a0, b0);
    rope_pair(x1, y1, c[2 * w + 1], s[2 * w + 1], a1, b1);
    xw[w] = Pack<BF16>::pack(a0, a1);
    yw[w] = Pack<BF16>::pack(b0, b1);
  }
}

// Interleaved pairing: rotate the 4 pairs (2k, 2k+1) held in one 16-byte chunk, pair w of the chunk
// with cos/sin c[w], s[w] (same arithmetic per pair as rope_pair).
template <bool BF16>
__device__ __forceinline__ void rope_rotate_chunk_il(uint4& v, const float* c, const float* s) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float e, o, a, b;
    Pack<BF16>::unpack(w[j], e, o);
    rope_pair(e, o, c[j], s[j], a, b);
    w[j] = Pack<BF16>::pack(a, b);
  }
}

// ---- packed form: cos/sin of 8 consecutive frequencies as 4 fp32 pairs --------------------------

struct RopeCS8 {
  uint64_t c[4], s[4];
};

// Exact cos/sin of pos * theta_k for k = k0 .. k0 + 7; lo/hi point at the F_k words (any memory
// space; kernels pass a shared-memory copy so per-lane indices do not serialise constant loads).
__device__ __forceinline__ void rope_cs8_exact(uint32_t pos, const uint32_t* lo, const uint32_t* hi, int k0,
                                               RopeCS8& o) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float c0, s0, c1, s1;
    rope_cs(pos, lo[k0 + 2 * j], hi[k0 + 2 * j], c0, s0);
    rope_cs(pos, lo[k0 + 2 * j + 1], hi[k0 + 2 * j + 1], c1, s1);
    o.c[j] = ptx::f2_pack(c0, c1);
    o.s[j] = ptx::f2_pack(s0, s1);
  }
}

// rope_cs8_exact for a signed position.
__device__ __forceinline__ void rope_cs8_exact_signed(int32_t pos, const uint32_t* lo, const uint32_t* hi, int k0,
                                                      RopeCS8& o) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float c0, s0, c1, s1;
    rope_cs_signed(pos, lo[k0 + 2 * j], hi[k0 + 2 * j], c0, s0);
    rope_cs_signed(pos, lo[k0 + 2 * j + 1], hi[k0 + 2 * j + 1], c1, s1);
    o.c[j] = ptx::f2_pack(c0, c1);
    o.s[j] = ptx::f2_pack(s0, s1);
  }
}

// a <- a * b as unit complex numbers (angle addition), same rounding as rope_advance per lane.
__device__ __forceinline__ void rope_cs8_advance(RopeCS8& a, const RopeCS8& b) {
  const uint64_t zero = ptx::f2_pack(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t cn = ptx::f2_fma(a.c[j], b.c[j], ptx::f2_mul(a.s[j], ptx::f2_sub(zero, b.s[j])));
    const uint64_t sn = ptx::f2_fma(a.s[j], b.c[j], ptx::f2_mul(a.c[j], b.s[j]));
    a.c[j] = cn;
    a.s[j] = sn;
  }
}

template <bool BF16>
__device__ __forceinline__ uint64_t unpack2(uint32_t w) {
  float lo, hi;
  Pack<BF16>::unpack(w, lo, hi);
  return ptx::f2_pack(lo, hi);
}

// Same rotation as rope_rotate_chunk (bit-identical per element for equal cos/sin), on fp32 pairs:
// x' = fma(x, c, y * (-s)), y' = fma(y, c, x * s).
template <bool BF16>
__device__ __forceinline__ void rope_rotate_chunk_cs8(uint4& xv, uint4& yv, const RopeCS8& cs) {
  uint32_t* xw = reinterpret_cast<uint32_t*>(&xv);
  uint32_t* yw = reinterpret_cast<uint32_t*>(&yv);
  const uint64_t zero = ptx::f2_pack(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t x = unpack2<BF16>(xw[j]);
    const uint64_t y = unpack2<BF16>(yw[j]);
    const uint64_t xr = ptx::f2_fma(x, cs.c[j], ptx::f2_mul(y, ptx::f2_sub(zero, cs.s[j])));
    const uint64_t yr = ptx::f2_fma(y, cs.c[j], ptx::f2_mul(x, cs.s[j]));
    float a0, a1, b0, b1;
    ptx::f2_unpack(xr, a0, a1);
    ptx::f2_unpack(yr, b0, b1);
    xw[j] = Pack<BF16>::pack(a0, a1);
    yw[j] = Pack<BF16>::pack(b0, b1);
  }
}

// Interleaved pairing with carried cos/sin: chunk `half` (0 or 1) of the thread's two adjacent
// chunks holds the pairs of frequencies 4 half .. 4 half + 3 of cs.
template <bool BF16>
__device__ __forceinline__ void rope_rotate_chunk_il_cs8(uint4& v, const RopeCS8& cs, int half) {
  float c[4], s[4];
  ptx::f2_unpack(cs.c[2 * half], c[0], c[1]);
  ptx::f2_unpack(cs.c[2 * half + 1], c[2], c[3]);
  ptx::f2_unpack(cs.s[2 * half], s[0], s[1]);
  ptx::f2_unpack(cs.s[2 * half + 1], s[2], s[3]);
  rope_rotate_chunk_il<BF16>(v, c, s);
}

}  // namespace attnfuse
