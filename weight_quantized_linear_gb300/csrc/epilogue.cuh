// epilogue.cuh -- optional terms of the int8 / fp8 GEMM's epilogue ("LMDeploy W8A8 quantisation
// guide", inference kernels: the _linear_add variant of matmul_kernel_dynamic_quant fuses a bias and
// a residual into c = c * rms_scale * linear_scale).  The sum is taken in fp32, left to right, after
// the scaled value and before the single rounding to fp16:
//     y[m, n] = fp16(((acc * xs[m]) * ws[n] + bias[n]) + residual[m, n])
// A null pointer leaves its term out (adding 0.0 would turn a -0.0 result into +0.0).
//
// The kernels load the terms they need ahead of their stores (a chunk of residual values at a time),
// so that the loads overlap; y may be the residual buffer itself, since each thread reads its own
// elements before it writes them.
#pragma once

#include <cuda_fp16.h>

namespace wql {

struct EpilogueAdd {
  const __half* bias;      // [N], or null
  const __half* residual;  // [M, N] row-major, or null; may be the output y itself
};

// u + b + r with the terms already widened to fp32; a term whose pointer is null is not added.
__device__ __forceinline__ float add_terms(float u, const EpilogueAdd& ea, float b, float r) {
  if (ea.bias) u = __fadd_rn(u, b);
  if (ea.residual) u = __fadd_rn(u, r);
  return u;
}

// Four consecutive fp16 values (8-byte aligned) widened to fp32.
__device__ __forceinline__ void load_half4(const __half* p, float (&v)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  const __half2 lo = *reinterpret_cast<const __half2*>(&raw.x), hi = *reinterpret_cast<const __half2*>(&raw.y);
  v[0] = __low2float(lo);
  v[1] = __high2float(lo);
  v[2] = __low2float(hi);
  v[3] = __high2float(hi);
}

}  // namespace wql
