// Device arithmetic shared by the selection kernels and the tensor-core
// router's fused selection epilogue.
#pragma once

#include <cuda_runtime.h>

namespace moe {

// Phi(u), the standard normal CDF, as erfc(-u / sqrt 2) / 2. erfc(z), z >= 0,
// is the Chebyshev-fitted form of Numerical Recipes (Press et al., 2nd ed.,
// section 6.2, "erfcc"): t exp(-z^2 + P(t)), t = 1 / (1 + z/2), P of degree 9,
// fractional error below 1.2e-7 for every z; erfc(-z) = 2 - erfc(z). In fp32,
// with z^2 compensated and the fast exponential, the relative error is about
// 1e-6 wherever Phi > 1e-7, far inside the tolerance of the balancing sums.
__device__ __forceinline__ float normal_cdf(float u) {
  const float w = -u * 0.70710678118654752f;
  const float z = fabsf(w);
  const float t = __fdividef(1.f, fmaf(0.5f, z, 1.f));
  float p = 0.17087277f;
  p = fmaf(t, p, -0.82215223f);
  p = fmaf(t, p, 1.48851587f);
  p = fmaf(t, p, -1.13520398f);
  p = fmaf(t, p, 0.27886807f);
  p = fmaf(t, p, -0.18628806f);
  p = fmaf(t, p, 0.09678418f);
  p = fmaf(t, p, 0.37409196f);
  p = fmaf(t, p, 1.00002368f);
  p = fmaf(t, p, -1.26551223f);
  const float zz = z * z;
  const float ez = fmaf(z, z, -zz);  // z^2 = zz + ez exactly
  const float half_erfc = 0.5f * t * __expf((p - zz) - ez);
  return w >= 0.f ? half_erfc : 1.f - half_erfc;
}

}  // namespace moe
