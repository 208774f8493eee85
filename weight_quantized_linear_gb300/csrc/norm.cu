// norm.cu -- QRMSNorm fused with per-token dynamic int8 quantisation, and the calibration
// statistic used by weight smoothing ("LMDeploy W8A8 quantisation guide": QRMSNorm.forward,
// rms_norm_dynamic_quant, per_token_quant_int8 with scale = absmax / 127 and codes rounded to
// integers; smoothing statistics are the per-channel absmax of the norm output).
//
// One CTA of 256 threads per token row.  The row is read once with 16-byte loads and kept in
// registers; the sum of squares uses a fixed order (chunk c of 8 elements belongs to thread
// c mod 256, which adds its elements in increasing k; the 256 partial sums are then folded
// pairwise (t, t+128), (t, t+64), ..., (t, t+1)), so int8 codes are reproducible bit for bit.
// Every float operation uses an explicitly rounded intrinsic: nothing is contracted into FMA.
#include "common.cuh"
#include "internal.h"

namespace wql {
namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ float block_sum_fixed(float p, float* red) {
  const int tid = threadIdx.x;
  red[tid] = p;
  __syncthreads();
#pragma unroll
  for (int s = 128; s >= 32; s >>= 1) {
    if (tid < s) red[tid] = __fadd_rn(red[tid], red[tid + s]);
    __syncthreads();
  }
  float total = 0.f;
  if (tid < 32) {
    float v = red[tid];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
    total = v;
  }
  if (tid == 0) red[256] = total;
  __syncthreads();
  total = red[256];
  __syncthreads();
  return total;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < kNormThreads / 32; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  return m;
}

// MODE 0: quantise (q, xs); MODE 1: per-channel absmax of the norm output (atomic max into absmax).
template <int CPT, int MODE>
__global__ void __launch_bounds__(kNormThreads)
    qrmsnorm_kernel(const __half* __restrict__ x, const __half* __restrict__ gamma, float eps, int K,
                    int8_t* __restrict__ q, float* __restrict__ xs, float* __restrict__ absmax) {
  __shared__ float red[260];
  const int m = blockIdx.x, tid = threadIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)m * K);
  const int nchunks = K >> 3;

  uint4 xv[CPT];
  float p = 0.f;
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int c = tid + kNormThreads * i;
    if (c < nchunks) {
      xv[i] = __ldg(xr + c);
      const __half* h = reinterpret_cast<const __half*>(&xv[i]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float v = __half2float(h[e]);
        p = __fadd_rn(p, __fmul_rn(v, v));
      }
    }
  }
  const float ss = block_sum_fixed(p, red);
  const float mean = __fdiv_rn(ss, (float)K);
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));

  float yv[CPT][8];
  float amax = 0.f;
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int c = tid + kNormThreads * i;
    if (c < nchunks) {
      const uint4 gv = __ldg(gr + c);
      const __half* h = reinterpret_cast<const __half*>(&xv[i]);
      const __half* gh = reinterpret_cast<const __half*>(&gv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float yy = __fmul_rn(__fmul_rn(__half2float(h[e]), r), __half2float(gh[e]));
        yv[i][e] = yy;
        amax = fmaxf(amax, fabsf(yy));
      }
    }
  }

  if (MODE == 1) {
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = tid + kNormThreads * i;
      if (c < nchunks) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          atomicMax(reinterpret_cast<int*>(absmax) + 8 * c + e, __float_as_int(fabsf(yv[i][e])));
      }
    }
    return;
  }

  const float rowmax = block_max(amax, red);
  const float scale = rowmax == 0.f ? 1.0f : __fdiv_rn(rowmax, 127.0f);
  if (tid == 0) xs[m] = scale;
  int8_t* qr = q + (size_t)m * K;
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int c = tid + kNormThreads * i;
    if (c < nchunks) {
      uint32_t packed[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float v = rintf(__fdiv_rn(yv[i][e], scale));
        v = fminf(fmaxf(v, -128.f), 127.f);
        packed[e >> 2] |= (uint32_t)(uint8_t)(int8_t)(int)v << (8 * (e & 3));
      }
      *reinterpret_cast<uint2*>(qr + 8 * c) = make_uint2(packed[0], packed[1]);
    }
  }
}

template <int MODE>
cudaError_t launch_norm(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K, int8_t* q, float* xs,
                        float* absmax, cudaStream_t s) {
  const __half* xh = reinterpret_cast<const __half*>(x);
  const __half* gh = reinterpret_cast<const __half*>(gamma);
  const int cpt = (K + 2047) / 2048;
  dim3 grid(M), block(kNormThreads);
  if (cpt <= 1)
    qrmsnorm_kernel<1, MODE><<<grid, block, 0, s>>>(xh, gh, eps, K, q, xs, absmax);
  else if (cpt <= 2)
    qrmsnorm_kernel<2, MODE><<<grid, block, 0, s>>>(xh, gh, eps, K, q, xs, absmax);
  else if (cpt <= 4)
    qrmsnorm_kernel<4, MODE><<<grid, block, 0, s>>>(xh, gh, eps, K, q, xs, absmax);
  else
    qrmsnorm_kernel<8, MODE><<<grid, block, 0, s>>>(xh, gh, eps, K, q, xs, absmax);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qrmsnorm_quant_i8(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K, int8_t* q,
                                     float* xs, cudaStream_t s) {
  return launch_norm<0>(x, gamma, eps, M, K, q, xs, nullptr, s);
}

cudaError_t launch_act_absmax(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K, float* absmax,
                              cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(absmax, 0, sizeof(float) * (size_t)K, s);
  if (e != cudaSuccess) return e;
  if (M == 0) return cudaSuccess;
  return launch_norm<1>(x, gamma, eps, M, K, nullptr, nullptr, absmax, s);
}

}  // namespace wql
