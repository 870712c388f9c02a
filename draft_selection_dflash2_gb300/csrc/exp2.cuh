// exp2.cuh -- 2^x for x <= 0 in fp32 with every step a correctly rounded IEEE
// operation, so that the walk's draws and verification's fixed-point weights
// are reproducible by any implementation of the same steps.
//
// Cody and Waite's range reduction (Software Manual for the Elementary
// Functions, 1980): x = n + f, n = rint(x), f in [-1/2, 1/2]; 2^f = e^(f ln 2)
// by the degree-7 Taylor polynomial, coefficients (ln 2)^k / k! rounded to
// fp32, in Horner form with fused multiply-adds; then an exact scaling by 2^n
// (correctly rounded when the result is subnormal).  0 below -126 and for NaN.
// The truncation error (f ln 2)^8 / 8! < 4e-10 is below half an fp32 ulp.
#pragma once

namespace dflash2 {

__device__ __forceinline__ float exp2_neg(float x) {
  if (!(x >= -126.0f)) return 0.0f;
  const float n = rintf(x);
  const float f = __fsub_rn(x, n);
  float p = 1.525273365e-05f;
  p = __fmaf_rn(p, f, 1.540352969e-04f);
  p = __fmaf_rn(p, f, 1.333355787e-03f);
  p = __fmaf_rn(p, f, 9.618128650e-03f);
  p = __fmaf_rn(p, f, 5.550410971e-02f);
  p = __fmaf_rn(p, f, 2.402265072e-01f);
  p = __fmaf_rn(p, f, 6.931471825e-01f);
  p = __fmaf_rn(p, f, 1.0f);
  return __fmul_rn(p, __int_as_float((static_cast<int>(n) + 127) << 23));
}

}  // namespace dflash2
