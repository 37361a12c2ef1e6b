// quant_common.cuh -- device helpers shared by the quantizers: streaming
// loads, bf16x2 absolute maxima, the E4M3 element map and warp maxima.
#pragma once

#include "fp_exact.cuh"
#include "internal.h"

namespace fp8rl {
namespace {

using fx::ScaleDiv;
using fx::make_scale_div;
using fx::scaled_quotient;

// ------------------------------------------------------------ device bits --

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// max |x| over the 8 bf16 of a 16-byte vector, folded into a bf16x2 running max
__device__ __forceinline__ uint32_t absmax8(uint32_t m, const uint4& v) {
  m = bf16x2_max(m, v.x & 0x7FFF7FFFu);
  m = bf16x2_max(m, v.y & 0x7FFF7FFFu);
  m = bf16x2_max(m, v.z & 0x7FFF7FFFu);
  m = bf16x2_max(m, v.w & 0x7FFF7FFFu);
  return m;
}

__device__ __forceinline__ float bf16x2_maxf(uint32_t m) {
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

// two binary32 -> two E4M3 codes (lo in the low byte), RNE, saturating
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// the element map over one bf16x2 word -> 2 codes
template <bool kGuard>
__device__ __forceinline__ uint32_t quant2(uint32_t w, const ScaleDiv& sd) {
  float x0 = __uint_as_float(w << 16);
  float x1 = __uint_as_float(w & 0xFFFF0000u);
  return cvt_e4m3x2(scaled_quotient<kGuard>(x0, sd), scaled_quotient<kGuard>(x1, sd));
}

// 8 bf16 -> 8 codes packed in a uint2 (any prepared scale)
template <bool kGuard>
__device__ __forceinline__ uint2 quant8(const uint4& v, const ScaleDiv& sd) {
  uint2 r;
  r.x = quant2<kGuard>(v.x, sd) | (quant2<kGuard>(v.y, sd) << 16);
  r.y = quant2<kGuard>(v.z, sd) | (quant2<kGuard>(v.w, sd) << 16);
  return r;
}

// The same for a scale known to be in the Markstein range (mode 1), with no
// per-element branch; kGuard as in scaled_quotient.
template <bool kGuard>
__device__ __forceinline__ float fast_quotient(float x, float s, float y) {
  float q = fx::markstein_quotient(x, s, y);
  if (kGuard) {
    const float q0 = __fmul_rn(x, y);
    q = fabsf(q0) < 1024.0f ? q : q0;
  }
  return q;
}
template <bool kGuard>
__device__ __forceinline__ uint32_t quant2_fast(uint32_t w, float s, float y) {
  return cvt_e4m3x2(fast_quotient<kGuard>(__uint_as_float(w << 16), s, y),
                    fast_quotient<kGuard>(__uint_as_float(w & 0xFFFF0000u), s, y));
}
template <bool kGuard>
__device__ __forceinline__ uint2 quant8_fast(const uint4& v, float s, float y) {
  uint2 r;
  r.x = quant2_fast<kGuard>(v.x, s, y) | (quant2_fast<kGuard>(v.y, s, y) << 16);
  r.y = quant2_fast<kGuard>(v.z, s, y) | (quant2_fast<kGuard>(v.w, s, y) << 16);
  return r;
}

// Dispatch once per scale: the common (mode 1) path has no element branch.
template <bool kGuard>
__device__ __forceinline__ uint2 quant8_any(const uint4& v, const ScaleDiv& sd) {
  return sd.mode == 1 ? quant8_fast<kGuard>(v, sd.s, sd.y) : quant8<kGuard>(v, sd);
}

__device__ __forceinline__ float warp_max(float v, int width) {
  for (int o = width >> 1; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

}  // namespace
}  // namespace fp8rl
