// 2^x on the FMA pipe, for moving part of a softmax's exponentials off the
// special-function unit (which issues 16 results per SM per clock, against
// 128 FMAs).
//
// Method: Cody-Waite range reduction x = j + f with j = round(x) obtained by
// the 1.5 * 2^23 shifter (adding it leaves j in the low mantissa bits, so the
// exponent of the result is formed with one integer add), and a degree-3
// polynomial for 2^f on [-1/2, 1/2].  The coefficients are this project's own
// fit: iterated weighted least squares on the relative error over a dense
// grid, converging to near-equal ripple; max relative error 7.5e-5 in fp32
// Horner evaluation, far below the bf16 rounding (2^-9) that P and dS undergo
// before the MMA.  Inputs below -126 are clamped (the result is then about
// 1.2e-38, not 0; callers that need an exact zero mask explicitly).
#pragma once
#include <cstdint>

namespace detattn {

__device__ __forceinline__ float exp2_poly(float x) {
  constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
  constexpr float c0 = 0.9999281167984009f;
  constexpr float c1 = 0.6932609677314758f;
  constexpr float c2 = 0.242610901594162f;
  constexpr float c3 = 0.05517147481441498f;
  x = fmaxf(x, -126.0f);
  const float t = x + kShift;
  const float f = x - (t - kShift);
  const float p = fmaf(fmaf(fmaf(c3, f, c2), f, c1), f, c0);
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

// ---- packed pairs: two fp32 lanes per 64-bit register, processed by the
// f32x2 FMA/add instructions (one issue slot for two results).
__device__ __forceinline__ uint64_t f2_make(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// exp2_poly on a pair, the floating-point steps done as f32x2 operations.
// Same method, coefficients and clamp as exp2_poly; results are identical.
__device__ __forceinline__ void exp2_poly2(float x0, float x1, float& y0, float& y1) {
  constexpr float kShift = 12582912.0f;
  x0 = fmaxf(x0, -126.0f);
  x1 = fmaxf(x1, -126.0f);
  const uint64_t x = f2_make(x0, x1);
  const uint64_t t = f2_add(x, f2_make(kShift, kShift));
  const uint64_t j = f2_add(t, f2_make(-kShift, -kShift));
  const uint64_t f = f2_fma(j, f2_make(-1.0f, -1.0f), x);
  uint64_t p = f2_fma(f2_make(0.05517147481441498f, 0.05517147481441498f), f,
                      f2_make(0.242610901594162f, 0.242610901594162f));
  p = f2_fma(p, f, f2_make(0.6932609677314758f, 0.6932609677314758f));
  p = f2_fma(p, f, f2_make(0.9999281167984009f, 0.9999281167984009f));
  float p0, p1, t0, t1;
  f2_split(p, p0, p1);
  f2_split(t, t0, t1);
  y0 = __int_as_float(__float_as_int(p0) + (__float_as_int(t0) << 23));
  y1 = __int_as_float(__float_as_int(p1) + (__float_as_int(t1) << 23));
}

}  // namespace detattn
