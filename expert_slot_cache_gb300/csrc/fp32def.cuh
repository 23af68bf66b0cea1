// fp32 functions defined operation by operation, so that a value built on them
// (a routing score, an 8-bit code) is reproducible bit for bit off the GPU.
#pragma once

#include <math.h>

namespace moe {

// exp: Cody and Waite's reduction n = rint(x log2 e), r = (x - n LN2_HI) -
// n LN2_LO (n LN2_HI exact), the degree-7 Taylor polynomial of e^r in Horner
// form, times 2^n.  Every step is one IEEE fp32 multiply, add or subtract (the
// _rn intrinsics keep the compiler from fusing them).  +inf above 88, 0 below
// -80 (2^n stays normal in between).
__device__ __forceinline__ float exp32_def(float x) {
  if (x > 88.f) return INFINITY;
  if (x < -80.f) return 0.f;
  const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));
  float r = __fsub_rn(x, __fmul_rn(n, 0x1.63p-1f));
  r = __fsub_rn(r, __fmul_rn(n, -0x1.bd0106p-13f));
  float p = 0x1.a01a02p-13f;
  p = __fadd_rn(__fmul_rn(p, r), 0x1.6c16c2p-10f);
  p = __fadd_rn(__fmul_rn(p, r), 0x1.111112p-7f);
  p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-5f);
  p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-3f);
  p = __fadd_rn(__fmul_rn(p, r), 0x1p-1f);
  p = __fadd_rn(__fmul_rn(p, r), 1.f);
  p = __fadd_rn(__fmul_rn(p, r), 1.f);
  return __fmul_rn(p, __int_as_float(((int)n + 127) << 23));
}

// sigmoid(l) = 1 / (1 + exp32(-l)): one IEEE add and one IEEE divide.
__device__ __forceinline__ float sigmoid32_def(float l) { return __fdiv_rn(1.f, __fadd_rn(1.f, exp32_def(-l))); }

// silu(g) = g / (1 + exp32(-g)).
__device__ __forceinline__ float silu32_def(float g) { return __fdiv_rn(g, __fadd_rn(1.f, exp32_def(-g))); }

// Symmetric 8-bit code of v for scale s (s = amax / 127): rint(v / s) clamped
// to [-127, 127]; 0 when s == 0.
__device__ __forceinline__ int q8_code(float v, float s) {
  if (!(s > 0.f)) return 0;
  const float q = rintf(__fdiv_rn(v, s));
  return (int)fminf(127.f, fmaxf(-127.f, q));
}

}  // namespace moe
