// swe_fastmath.cuh -- double-precision reciprocal and reciprocal square root
// for GB300, whose FP64 pipe is narrow: a hardware approximation refined by
// Newton-Raphson iterations (Newton's method on f(y) = 1/y - x and on
// f(y) = 1/y^2 - x), in place of the correctly rounded library routines.
//
// The seeds are the PTX instructions rcp.approx.ftz.f64 and
// rsqrt.approx.ftz.f64 (about 20 correct bits); each iteration roughly doubles
// the number of correct bits, so two give the full 53-bit significand up to
// about one unit in the last place (checked against 1/x and 1/sqrt(x) on the
// GPU by the test suite).  Non-positive, non-finite or subnormal arguments
// give a non-finite result (the kernels report those states as errors).
#pragma once

#include <cuda_runtime.h>

namespace swe {

__device__ __forceinline__ double rcp_nr(double x) {
  double y;
  asm("rcp.approx.ftz.f64 %0, %1;" : "=d"(y) : "d"(x));
  // y <- y + y (1 - x y), twice
  double e = fma(-x, y, 1.0);
  y = fma(y, e, y);
  e = fma(-x, y, 1.0);
  return fma(y, e, y);
}

__device__ __forceinline__ double rsq_nr(double x) {
  double y;
  asm("rsqrt.approx.ftz.f64 %0, %1;" : "=d"(y) : "d"(x));
  // y <- y + (y / 2) (1 - x y^2), twice
  double e = fma(-x * y, y, 1.0);
  y = fma(0.5 * y, e, y);
  e = fma(-x * y, y, 1.0);
  return fma(0.5 * y, e, y);
}

}  // namespace swe
