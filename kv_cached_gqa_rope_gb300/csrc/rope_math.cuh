// Split-half RoPE arithmetic shared by the store kernel (K1) and the fused
// decode step (K2 in single-launch mode).  Internal to libkvgqa.
//
// microLLM-rocm ARCHITECTURE.md, section "Attention layout boundary":
// split-half RoPE needs an even head width, a nonnegative position and a
// positive base.  Pair i is (x[i], x[i + D/2]) at angle pos * theta^(-2i/D).
#pragma once

#include <cstdint>

namespace kvgqa {

struct __align__(16) CosSin {
  float ch, cl, sh, sl;  // cos = ch + cl, sin = sh + sl
};

// ---------------------------------------------------------------- double-float
// A value held as an unevaluated sum h + l of two FP32 numbers (|l| <= ulp(h)/2),
// with the error-free sum of Knuth and the FMA-based exact product (Dekker's
// double-length arithmetic).  Intrinsics keep the compiler from contracting
// or reordering the error terms.
struct DF {
  float h, l;
};

__device__ __forceinline__ DF df_fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return DF{s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ DF df_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return DF{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const DF s = df_two_sum(a.h, b.h);
  return df_fast_two_sum(s.h, __fadd_rn(s.l, __fadd_rn(a.l, b.l)));
}
__device__ __forceinline__ DF df_add_f(DF a, float b) {
  const DF s = df_two_sum(a.h, b);
  return df_fast_two_sum(s.h, __fadd_rn(s.l, a.l));
}
__device__ __forceinline__ DF df_mul(DF a, DF b) {
  const float p = __fmul_rn(a.h, b.h);
  float e = __fmaf_rn(a.h, b.h, -p);  // the product's rounding error, exactly
  e = __fmaf_rn(a.h, b.l, e);
  e = __fmaf_rn(a.l, b.h, e);
  return df_fast_two_sum(p, e);
}
// A double as a double-float (both parts computed in FP64, then rounded).
__host__ __device__ constexpr DF df_const(double v) {
  return DF{static_cast<float>(v), static_cast<float>(v - static_cast<double>(static_cast<float>(v)))};
}

// cos and sin of pos * f, f one of the RoPE frequencies given as f * 2/pi
// (quarter turns per position step: fraction `frac` in 64-bit fixed point,
// integer part mod 4 `quad`), as FP32 hi+lo pairs with an absolute error of
// a few 1e-14.  The reduction modulo pi/2 is Payne and Hanek's: with the
// frequency already scaled by 2/pi to 64 fractional bits, pos * f in quarter
// turns is an exact integer product (a position is below 2^31), whose upper
// bits count whole quarter turns and whose lower 64 bits are the fraction.
// Rounding to the nearest quarter turn leaves a signed fraction of at most
// one half, which becomes the reduced angle |x| <= pi/4 as a double-float
// (its top 48 bits, exactly, times pi/2 * 2^-48).  The reduction thus costs a
// few integer operations instead of FP64 arithmetic, which runs at a small
// fraction of the FP32 rate on this GPU.  sin x and cos x are then Taylor
// series (coefficients 1/n!) evaluated in double-float FP32 arithmetic by
// Horner's rule: the terms up to x^5 (sin) and x^6 (cos) in double-float, the
// smaller ones (below 4e-5 in size) in plain FP32; the first omitted terms,
// x^15/15! and x^14/14!, are below 3e-14 for |x| <= pi/4.  The quadrant then
// maps (sin x, cos x) to (sin, cos) of the whole angle.
__device__ __forceinline__ CosSin rope_cos_sin(int pos, uint64_t frac, uint32_t quad) {
  const uint32_t n = static_cast<uint32_t>(pos);  // 0 <= pos < 2^31
  const uint64_t lo = static_cast<uint64_t>(n) * static_cast<uint32_t>(frac);
  const uint64_t hi = static_cast<uint64_t>(n) * static_cast<uint32_t>(frac >> 32);
  const uint64_t f64 = lo + (hi << 32);  // n * frac mod 2^64: the fraction of a quarter turn
  const uint32_t whole = static_cast<uint32_t>(hi >> 32) + (f64 < lo ? 1u : 0u) + n * quad;
  // a fraction of one half or more rounds up to the next quarter turn, and
  // its signed reading (f64 - 2^64) is then the remainder
  const uint32_t q = (whole + static_cast<uint32_t>(f64 >> 63)) & 3u;
  const int64_t r = static_cast<int64_t>(f64) >> 16;  // |r| <= 2^47, units of 2^-48 quarter turns
  const DF rd = df_two_sum(static_cast<float>(static_cast<int32_t>(r >> 24)) * 16777216.0f,  // both exact
                           static_cast<float>(static_cast<int32_t>(r & 0xffffff)));
  constexpr DF kQuarterTurn48 = df_const(1.5707963267948966 / 281474976710656.0);  // pi/2 * 2^-48
  const DF x = df_mul(rd, kQuarterTurn48);
  const DF y = df_mul(x, x);  // x^2
  // sin x = x (1 + y (-1/3! + y (1/5! + y Ts))), Ts = -1/7! + y/9! - y^2/11! + y^3/13!
  const float ts = __fmaf_rn(__fmaf_rn(__fmaf_rn(y.h, 1.0f / 6227020800.0f, -1.0f / 39916800.0f), y.h,
                                       1.0f / 362880.0f),
                             y.h, -1.0f / 5040.0f);
  const DF s3 = df_add_f(df_const(1.0 / 120.0), __fmul_rn(y.h, ts));
  const DF s2 = df_add(df_const(-1.0 / 6.0), df_mul(y, s3));
  const DF s1 = df_add(df_const(1.0), df_mul(y, s2));
  const DF sx = df_mul(x, s1);
  // cos x = 1 + y (-1/2! + y (1/4! + y (-1/6! + y Tc))), Tc = 1/8! - y/10! + y^2/12!
  const float tc = __fmaf_rn(__fmaf_rn(y.h, 1.0f / 479001600.0f, -1.0f / 3628800.0f), y.h, 1.0f / 40320.0f);
  const DF c4 = df_add_f(df_const(-1.0 / 720.0), __fmul_rn(y.h, tc));
  const DF c3 = df_add(df_const(1.0 / 24.0), df_mul(y, c4));
  const DF c2 = df_add(df_const(-0.5), df_mul(y, c3));
  const DF cx = df_add(df_const(1.0), df_mul(y, c2));
  // the angle is x + q * pi/2
  DF c, s;
  switch (q) {
    case 0: c = cx; s = sx; break;
    case 1: c = DF{-sx.h, -sx.l}; s = cx; break;
    case 2: c = DF{-cx.h, -cx.l}; s = DF{-sx.h, -sx.l}; break;
    default: c = sx; s = DF{-cx.h, -cx.l}; break;
  }
  CosSin v;
  v.ch = c.h;
  v.cl = c.l;
  v.sh = s.h;
  v.sl = s.l;
  return v;
}

// x1 * C - x2 * S with C, S given as hi+lo pairs.  Products are split exactly
// with FMA; intrinsics keep the compiler from contracting them differently,
// so the BF16 result is one rounding of an almost exact value even where the
// difference cancels.
__device__ __forceinline__ float rot_first(float x1, float x2, const CosSin& cs) {
  const float p = __fmul_rn(x1, cs.ch);
  const float pe = __fmaf_rn(x1, cs.ch, -p);
  const float q = __fmul_rn(x2, cs.sh);
  const float qe = __fmaf_rn(x2, cs.sh, -q);
  const float lo = __fmaf_rn(x1, cs.cl, __fmaf_rn(-x2, cs.sl, __fsub_rn(pe, qe)));
  return __fadd_rn(__fsub_rn(p, q), lo);
}

// x2 * C + x1 * S.
__device__ __forceinline__ float rot_second(float x1, float x2, const CosSin& cs) {
  const float p = __fmul_rn(x2, cs.ch);
  const float pe = __fmaf_rn(x2, cs.ch, -p);
  const float q = __fmul_rn(x1, cs.sh);
  const float qe = __fmaf_rn(x1, cs.sh, -q);
  const float lo = __fmaf_rn(x2, cs.cl, __fmaf_rn(x1, cs.sl, __fadd_rn(pe, qe)));
  return __fadd_rn(__fadd_rn(p, q), lo);
}

}  // namespace kvgqa
