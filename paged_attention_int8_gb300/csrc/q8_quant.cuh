// q8 arithmetic shared by the store kernels (kv_store.cu, kv_store_rope.cu):
// the group scale and the exact code of a value near a rounding tie.
//
// q8 ("shared/attention_kit.py", quantize_q8): per group of 32 channels
// s = max(max|x| / 127, 1e-8) in fp32, code = clamp(round_half_away(x / s),
// -127, 127) of the IEEE fp32 quotient.
#pragma once

#include "common.cuh"

namespace paq8 {

// fp32 group scale from the group's max |x|: max(amax / 127, 1e-8).
__device__ __forceinline__ float group_scale(float amax) {
  const float s = __fdiv_rn(amax, 127.0f);
  return s < 1e-8f ? 1e-8f : s;
}

// Code of x near a rounding tie: round_half_away(Q) for the IEEE quotient
// Q = RN(x / s), decided without a divide.  t is the half-integer within
// 2^-15 of q = x * rs (so |x / s - t| < 2^-14); e = x - t * s is then exact
// in one FMA (its bits span fewer than 24 places), and sign(e) orders x / s
// against t.  Q == t exactly when x / s lies within half the fp32 spacing
// next to t (ties of that rounding go to t, whose significand is even), and
// then the code goes away from zero; otherwise Q lies on the side of t that
// x / s does.  Below |t| = 0.5, a power of two, the spacing halves.
__device__ __forceinline__ int32_t tie_code(float x, float s, float rs) {
  const float q = __fmul_rn(x, rs);
  const float at = floorf(fabsf(q)) + 0.5f;  // |t|
  const float t = copysignf(at, q);
  const float e = __fmaf_rn(-t, s, x);       // x - t * s, exact
  // half the spacing of fp32 numbers just below |t| (|t| >= 0.5)
  float half_gap = __uint_as_float((__float_as_uint(at) & 0x7f800000u) - (24u << 23));
  if (at == 0.5f) half_gap *= 0.5f;
  const bool beyond = e != 0.0f && ((e > 0.0f) == (q > 0.0f));  // |x / s| > |t|
  const bool away = e == 0.0f || beyond || fabsf(e) <= __fmul_rn(half_gap, s);
  const int32_t m = static_cast<int32_t>(at) + (away ? 1 : 0);  // |code|
  return q < 0.0f ? -m : m;
}

// The same rule from the half-integer h itself (x / s within 2^-14 of h),
// as the bits of code + 1.5 * 2^23, whose low byte is the code's two's
// complement byte: e = x - h * s is exact, RN(x / s) == h when |e| is at most
// half the spacing below |h| times s (the spacing of the float before |h|,
// so that |h| = 0.5 needs no special case), and the code is h moved half a
// step away from zero when RN(x / s) == h or x / s lies beyond h (e and h of
// one sign), else half a step toward zero.
__device__ __forceinline__ uint32_t tie_code_bits(float x, float s, float h) {
  const float e = __fmaf_rn(-h, s, x);
  const uint32_t hb = __float_as_uint(h);
  const float half_gap =
      __uint_as_float((((hb & 0x7fffffffu) - 1u) & 0x7f800000u) - (24u << 23));
  const bool away = fabsf(e) <= __fmul_rn(half_gap, s) ||
                    static_cast<int32_t>(__float_as_uint(e) ^ hb) >= 0;
  const float step = __uint_as_float((hb & 0x80000000u) | 0x3f000000u);  // copysign(0.5, h)
  const float code = __fadd_rn(h, away ? step : -step);
  return __float_as_uint(__fadd_rn(code, 12582912.0f));
}

}  // namespace paq8
