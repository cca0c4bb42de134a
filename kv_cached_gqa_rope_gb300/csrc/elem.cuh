// Storage element types of the path: BF16 (the default) and IEEE binary16
// (FP16 cached rows).  Values cross memory as 16-bit patterns; all arithmetic
// is FP32, and every stored result is rounded once, to nearest even, in the
// storage format.  Internal to libkvgqa.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace kvgqa {

template <bool F16>
struct Elem;

template <>
struct Elem<false> {  // BF16
  // Operand format code of tcgen05.mma kind::f16 (A and B must agree).
  static constexpr uint32_t kMmaFormat = 1;
  __device__ static __forceinline__ float to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
  __device__ static __forceinline__ uint16_t from_f32(float v) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<const uint16_t*>(&b);
  }
  // Two values packed in a 32-bit word (element 0 in the low half) <-> FP32.
  __device__ static __forceinline__ float2 pair_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  __device__ static __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
};

template <>
struct Elem<true> {  // IEEE binary16
  static constexpr uint32_t kMmaFormat = 0;
  __device__ static __forceinline__ float to_f32(uint16_t b) { return __half2float(__ushort_as_half(b)); }
  __device__ static __forceinline__ uint16_t from_f32(float v) { return __half_as_ushort(__float2half_rn(v)); }
  __device__ static __forceinline__ float2 pair_to_f2(uint32_t w) {
    const __half2 h = *reinterpret_cast<const __half2*>(&w);
    return __half22float2(h);
  }
  __device__ static __forceinline__ uint32_t pack2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
};

}  // namespace kvgqa
