// epilogue.cuh -- optional terms of the int8 GEMM's epilogue ("LMDeploy W8A8 quantisation guide",
// inference kernels: the _linear_add variant of matmul_kernel_dynamic_quant fuses a bias and a
// residual into c = c * rms_scale * linear_scale).  The sum is taken in fp32, left to right, after
// the scaled value and before the single rounding to fp16:
//     y[m, n] = fp16(((acc * xs[m]) * ws[n] + bias[n]) + residual[m, n])
// A null pointer leaves its term out (adding 0.0 would turn a -0.0 result into +0.0).
#pragma once

#include <cuda_fp16.h>

namespace wql {

struct EpilogueAdd {
  const __half* bias;      // [N], or null
  const __half* residual;  // [M, N] row-major, or null; may be the output y itself
};

__device__ __forceinline__ float epilogue_add(float u, const EpilogueAdd& ea, int m, int n, int N) {
  if (ea.bias) u = __fadd_rn(u, __half2float(ea.bias[n]));
  if (ea.residual) u = __fadd_rn(u, __half2float(ea.residual[(size_t)m * N + n]));
  return u;
}

}  // namespace wql
