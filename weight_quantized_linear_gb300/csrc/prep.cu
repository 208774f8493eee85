// prep.cu -- weight preparation kernels (run once per layer, not per token):
//   awq_pack           asymmetric per-group int4 quantisation + packing ("LMDeploy ... INT4
//                      quantisation" tutorial, section 2; "AUQ dual-process framework" article,
//                      sections 3.3 and 5.4 for the qweight / scales / zeros tensor set)
//   smooth             SmoothQuant smoothing with alpha = 0.5 ("LMDeploy W8A8 quantisation guide",
//                      weight smoothing: smooth_ln_fcs)
//   per_channel_quant  symmetric int8 per output channel with fp32 scales (same guide, QLinear /
//                      per_channel_quant)
// All arithmetic is fp32 with explicitly rounded intrinsics, round-half-to-even, so the packed
// codes, scales and zero points are reproducible bit for bit.
#include "common.cuh"
#include "internal.h"

namespace wql {
namespace {

__device__ __forceinline__ float clamp_rint(float v, float lo, float hi) {
  float r = rintf(v);
  r = fmaxf(r, lo);  // fmaxf(NaN, lo) = lo
  return fminf(r, hi);
}

// One thread per (group, packed word column): 8 output columns x G rows.
__global__ void __launch_bounds__(128)
    awq_pack_kernel(const float* __restrict__ w, int N, int G, uint32_t* __restrict__ qweight,
                    __half* __restrict__ scales, uint32_t* __restrict__ qzeros) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int g = blockIdx.y;
  const int NW = N >> 3;
  if (c >= NW) return;
  const int k0 = g * G;
  float mn[8], mx[8];
  {
    const float4* row = reinterpret_cast<const float4*>(w + (size_t)k0 * N + 8 * c);
    const float4 a = __ldg(row), b = __ldg(row + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) mn[e] = mx[e] = v[e];
  }
  for (int k = k0 + 1; k < k0 + G; ++k) {
    const float4* row = reinterpret_cast<const float4*>(w + (size_t)k * N + 8 * c);
    const float4 a = __ldg(row), b = __ldg(row + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      mn[e] = fminf(mn[e], v[e]);
      mx[e] = fmaxf(mx[e], v[e]);
    }
  }
  float s[8];
  uint32_t zword = 0u;
  __align__(16) __half sh[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    __half h = __float2half_rn(__fdiv_rn(__fsub_rn(mx[e], mn[e]), 15.0f));
    if ((__half_as_ushort(h) & 0x7fffu) == 0) h = __ushort_as_half(0x3c00u);
    sh[e] = h;
    s[e] = __half2float(h);
    const float z = clamp_rint(__fdiv_rn(-mn[e], s[e]), 0.f, 15.f);
    zword |= (uint32_t)z << (4 * e);
  }
  qzeros[(size_t)g * NW + c] = zword;
  *reinterpret_cast<uint4*>(scales + (size_t)g * N + 8 * c) = *reinterpret_cast<const uint4*>(sh);
  for (int k = k0; k < k0 + G; ++k) {
    const float4* row = reinterpret_cast<const float4*>(w + (size_t)k * N + 8 * c);
    const float4 a = __ldg(row), b = __ldg(row + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t word = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float zf = (float)((zword >> (4 * e)) & 15u);
      const float q = clamp_rint(__fadd_rn(rintf(__fdiv_rn(v[e], s[e])), zf), 0.f, 15.f);
      word |= (uint32_t)q << (4 * e);
    }
    qweight[(size_t)k * NW + c] = word;
  }
}

__device__ __forceinline__ float block_max256(float v, float* red) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  return m;
}

// One CTA per input channel j: w_j = max_n |w[j, n]|, s_j = sqrt(a_j / w_j), fold into gamma and w.
__global__ void __launch_bounds__(256)
    smooth_kernel(const float* __restrict__ absmax, const __half* __restrict__ gamma, const float* w, int N,
                  float* __restrict__ s_out, __half* __restrict__ gamma_out, float* w_out) {
  __shared__ float red[8];
  const int j = blockIdx.x;
  const float* wr = w + (size_t)j * N;
  float m = 0.f;
  for (int n = threadIdx.x; n < N; n += blockDim.x) m = fmaxf(m, fabsf(wr[n]));
  const float wmax = block_max256(m, red);
  const float a = absmax[j];
  const float s = (a > 0.f && wmax > 0.f) ? __fsqrt_rn(__fdiv_rn(a, wmax)) : 1.0f;
  if (threadIdx.x == 0) {
    s_out[j] = s;
    gamma_out[j] = __float2half_rn(__fdiv_rn(__half2float(gamma[j]), s));
  }
  float* wo = w_out + (size_t)j * N;
  for (int n = threadIdx.x; n < N; n += blockDim.x) wo[n] = __fmul_rn(wr[n], s);
}

// Per output column n: ws_n = max_k |w[k, n]| / 127.  Block (32, 8) covers 32 columns.
__global__ void __launch_bounds__(256)
    colmax_scale_kernel(const float* __restrict__ w, int K, int N, float* __restrict__ ws) {
  __shared__ float red[8][33];
  const int n = blockIdx.x * 32 + threadIdx.x;
  float m = 0.f;
  if (n < N)
    for (int k = threadIdx.y; k < K; k += 8) m = fmaxf(m, fabsf(w[(size_t)k * N + n]));
  red[threadIdx.y][threadIdx.x] = m;
  __syncthreads();
  if (threadIdx.y == 0 && n < N) {
    float a = red[0][threadIdx.x];
    for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i][threadIdx.x]);
    ws[n] = a == 0.f ? 1.0f : __fdiv_rn(a, 127.0f);
  }
}

// qw[n, k] = clamp(rint(w[k, n] / ws_n), -127, 127), transposed through a 32x32 shared tile.
__global__ void __launch_bounds__(256)
    quant_transpose_kernel(const float* __restrict__ w, const float* __restrict__ ws, int K, int N,
                           int8_t* __restrict__ qw) {
  __shared__ int8_t tile[32][36];
  const int n0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  const int n = n0 + threadIdx.x;
  const float scale = n < N ? ws[n] : 1.0f;
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int k = k0 + r;
    int8_t v = 0;
    if (k < K && n < N) v = (int8_t)(int)clamp_rint(__fdiv_rn(w[(size_t)k * N + n], scale), -127.f, 127.f);
    tile[threadIdx.x][r] = v;  // tile[col][row]
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int nn = n0 + r, kk = k0 + threadIdx.x;
    if (nn < N && kk < K) qw[(size_t)nn * K + kk] = tile[r][threadIdx.x];
  }
}

}  // namespace

cudaError_t launch_awq_pack(const float* w, int K, int N, int group, uint32_t* qweight, uint16_t* scales,
                            uint32_t* qzeros, cudaStream_t s) {
  const int NW = N / 8;
  dim3 block(128), grid((NW + 127) / 128, K / group);
  awq_pack_kernel<<<grid, block, 0, s>>>(w, N, group, qweight, reinterpret_cast<__half*>(scales), qzeros);
  return cudaGetLastError();
}

cudaError_t launch_smooth(const float* absmax, const uint16_t* gamma, const float* w, int K, int N, float* s_out,
                          uint16_t* gamma_out, float* w_out, cudaStream_t s) {
  smooth_kernel<<<K, 256, 0, s>>>(absmax, reinterpret_cast<const __half*>(gamma), w, N, s_out,
                                  reinterpret_cast<__half*>(gamma_out), w_out);
  return cudaGetLastError();
}

cudaError_t launch_per_channel_quant_i8(const float* w, int K, int N, int8_t* qw, float* ws, cudaStream_t s) {
  colmax_scale_kernel<<<(N + 31) / 32, dim3(32, 8), 0, s>>>(w, K, N, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  quant_transpose_kernel<<<dim3((N + 31) / 32, (K + 31) / 32), dim3(32, 8), 0, s>>>(w, ws, K, N, qw);
  return cudaGetLastError();
}

}  // namespace wql
