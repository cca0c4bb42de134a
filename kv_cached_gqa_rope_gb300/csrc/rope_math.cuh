// Split-half RoPE arithmetic shared by the store kernel (K1) and the fused
// decode step (K2 in single-launch mode).  Internal to libkvgqa.
//
// microLLM-rocm ARCHITECTURE.md, section "Attention layout boundary":
// split-half RoPE needs an even head width, a nonnegative position and a
// positive base.  Pair i is (x[i], x[i + D/2]) at angle pos * theta^(-2i/D).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace kvgqa {

struct __align__(16) CosSin {
  float ch, cl, sh, sl;  // cos = ch + cl, sin = sh + sl
};

// cos and sin of pos * inv_freq, as FP32 hi+lo pairs.  The angle is formed
// in FP64 and reduced by 2*pi with a two-constant Cody-Waite step (2*pi split
// in two doubles, the products fused), so sincos only ever sees |r| <= pi.
__device__ __forceinline__ CosSin rope_cos_sin(int pos, double inv_freq) {
  constexpr double kTwoPiHi = 6.283185307179586232;    // nearest double to 2*pi
  constexpr double kTwoPiLo = 2.4492935982947064e-16;  // 2*pi - kTwoPiHi
  const double phi = static_cast<double>(pos) * inv_freq;
  const double k = rint(phi * 0.15915494309189535);    // 1 / (2*pi)
  const double r = fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, phi));
  double s, c;
  sincos(r, &s, &c);
  CosSin v;
  v.ch = static_cast<float>(c);
  v.cl = static_cast<float>(c - static_cast<double>(v.ch));
  v.sh = static_cast<float>(s);
  v.sl = static_cast<float>(s - static_cast<double>(v.sh));
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

__device__ __forceinline__ uint16_t bf16_rn_bits(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);  // round to nearest even
  return *reinterpret_cast<const uint16_t*>(&b);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

}  // namespace kvgqa
