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

// Sum of the 256 lane partials in the fixed order (t, t+128), (t, t+64), ..., (t, t+1).  The three
// cross-warp levels are evaluated by lane l of warp 0 from the eight partials l + 32 w, in exactly
// that order; the last five levels are warp shuffles.  Two barriers; every thread gets the total.
__device__ __forceinline__ float block_sum_fixed(float p, float* red) {
  const int tid = threadIdx.x;
  red[tid] = p;
  __syncthreads();
  if (tid < 32) {
    const float* r = red + tid;
    const float a0 = __fadd_rn(r[0], r[128]), a1 = __fadd_rn(r[64], r[192]);    // (t, t+128) at t, t+64
    const float a2 = __fadd_rn(r[32], r[160]), a3 = __fadd_rn(r[96], r[224]);   // ... at t+32, t+96
    const float b0 = __fadd_rn(a0, a1), b1 = __fadd_rn(a2, a3);                  // (t, t+64) at t, t+32
    float v = __fadd_rn(b0, b1);                                                 // (t, t+32)
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
    if (tid == 0) red[256] = v;
  }
  __syncthreads();
  return red[256];
}

// Row maximum; `slot` selects a scratch area distinct from the one the sum used, so one barrier
// suffices.
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  if ((threadIdx.x & 31) == 0) red[264 + (threadIdx.x >> 5)] = v;
  __syncthreads();
  float m = red[264];
#pragma unroll
  for (int w = 1; w < kNormThreads / 32; ++w) m = fmaxf(m, red[264 + w]);
  return m;
}

// round_half_even(fl(y / s)) clamped to [-128, 127], without a division in the common case.
// t = fl(y * inv) with inv = fl(1 / s) lies within 2.3e-5 of fl(y / s) when |y / s| <= 127.5
// (two roundings of relative size 2^-24 each, plus fl(y / s)'s own half ulp), so whenever t is
// more than 5e-5 away from a half-integer, both round to the same integer.  Otherwise the exact
// quotient is computed.
__device__ __forceinline__ float quant_code(float y, float s, float inv) {
  const float t = __fmul_rn(y, inv);
  const float fr = fabsf(t - truncf(t));  // distance above the lower integer, in [0, 1)
  float r;
  if (fabsf(fr - 0.5f) > 5e-5f) {
    r = rintf(t);
  } else {
    r = rintf(__fdiv_rn(y, s));
  }
  return fminf(fmaxf(r, -128.f), 127.f);
}

// MODE 0: quantise (q, xs); MODE 1: per-channel absmax of the norm output (atomic max into absmax).
// A CTA normalises R consecutive rows (R = 1 as launched); every row's 16-byte loads are issued
// before the first reduction.
template <int CPT, int R, int MODE>
__global__ void __launch_bounds__(kNormThreads)
    qrmsnorm_kernel(const __half* __restrict__ x, const __half* __restrict__ gamma, float eps, int M, int K,
                    int8_t* __restrict__ q, float* __restrict__ xs, float* __restrict__ absmax) {
  __shared__ float red[272];  // [0, 256) lane partials, 256 row sum, [264, 272) warp maxima
  const int tid = threadIdx.x;
  // programmatic dependent launch: the next kernel (typically the int8 GEMM) may start fetching its
  // weights now; this kernel's input comes from the preceding kernel
  if (tid == 0) grid_dependents_launch();
  grid_dependency_wait();
  const int nchunks = K >> 3;
  const int m0 = blockIdx.x * R;

  uint4 xv[R][CPT];
#pragma unroll
  for (int rr = 0; rr < R; ++rr) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)(m0 + rr) * K);
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = tid + kNormThreads * i;
      if (m0 + rr < M && c < nchunks) xv[rr][i] = __ldg(xr + c);
    }
  }

#pragma unroll
  for (int rr = 0; rr < R; ++rr) {
    const int m = m0 + rr;
    if (m >= M) break;  // uniform over the CTA
    float p = 0.f;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = tid + kNormThreads * i;
      if (c < nchunks) {
        const __half* h = reinterpret_cast<const __half*>(&xv[rr][i]);
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
        const __half* h = reinterpret_cast<const __half*>(&xv[rr][i]);
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
      continue;
    }

    const float rowmax = block_max(amax, red);
    const float scale = rowmax == 0.f ? 1.0f : __fdiv_rn(rowmax, 127.0f);
    const float inv = __fdiv_rn(1.0f, scale);
    if (tid == 0) xs[m] = scale;
    int8_t* qr = q + (size_t)m * K;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = tid + kNormThreads * i;
      if (c < nchunks) {
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float v = quant_code(yv[i][e], scale, inv);
          packed[e >> 2] |= (uint32_t)(uint8_t)(int8_t)(int)v << (8 * (e & 3));
        }
        *reinterpret_cast<uint2*>(qr + 8 * c) = make_uint2(packed[0], packed[1]);
      }
    }
  }
}

// Launch with programmatic stream serialisation: the kernel may start while its predecessor drains
// (it waits with griddepcontrol.wait before touching its inputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

template <int MODE>
cudaError_t launch_norm(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K, int8_t* q, float* xs,
                        float* absmax, cudaStream_t s) {
  const __half* xh = reinterpret_cast<const __half*>(x);
  const __half* gh = reinterpret_cast<const __half*>(gamma);
  const int cpt = (K + 2047) / 2048;
  // one row per CTA (two rows per CTA measured slower at M = 4096)
  const dim3 grid(M), block(kNormThreads);
  if (cpt <= 1) return launch_pdl(qrmsnorm_kernel<1, 1, MODE>, grid, block, s, xh, gh, eps, M, K, q, xs, absmax);
  if (cpt <= 2) return launch_pdl(qrmsnorm_kernel<2, 1, MODE>, grid, block, s, xh, gh, eps, M, K, q, xs, absmax);
  if (cpt <= 4) return launch_pdl(qrmsnorm_kernel<4, 1, MODE>, grid, block, s, xh, gh, eps, M, K, q, xs, absmax);
  return launch_pdl(qrmsnorm_kernel<8, 1, MODE>, grid, block, s, xh, gh, eps, M, K, q, xs, absmax);
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
