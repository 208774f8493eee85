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

// rint(x / s) for the correctly rounded quotient x / s, computed as x * (1 / s): the product is
// within 1.5 * 2^-23 of the quotient, relatively, so only a product closer than `margin` to a
// half-integer takes the exact division.  Beyond |x / s| = `limit` the callers clamp, and a
// difference of one in the rounded value does not change the clamped code.
__device__ __forceinline__ float rint_div(float x, float s, float inv, float limit, float margin) {
  const float t = __fmul_rn(x, inv);
  const float at = fabsf(t);
  if (at < limit && fabsf(__fsub_rn(__fsub_rn(at, truncf(at)), 0.5f)) < margin) return rintf(__fdiv_rn(x, s));
  return rintf(t);
}

// One CTA of 256 threads per (group, 1024 / G packed word columns).  Thread (slice, c) holds four
// consecutive output columns (one 16-byte load per row; half a packed word) for the kPackRows rows
// [slice kPackRows, (slice + 1) kPackRows) of the group in registers, so the weights are read from
// memory exactly once.  The G / kPackRows slices combine their minima / maxima in shared memory;
// every thread then derives the same scales and zero points, quantises the rows it holds, and the
// two threads of a word (adjacent lanes) join their nibbles with one shuffle.
constexpr int kPackRows = 8;
constexpr int kPackThreads = 256;

// Four CTAs per SM (64 registers, a 16-byte spill) measured faster than three without the cap:
// K = 4096, N = 11008, G = 128: 64.3 -> 60.0 us.
__global__ void __launch_bounds__(kPackThreads, 4)
    awq_pack_kernel(const float* __restrict__ w, int N, int G, uint32_t* __restrict__ qweight,
                    __half* __restrict__ scales, uint32_t* __restrict__ qzeros) {
  __shared__ float red_mn[4][kPackThreads + 8], red_mx[4][kPackThreads + 8];  // [element][thread]
  const int slices = G / kPackRows;        // 4, 8 or 16
  const int cols = kPackThreads / slices;  // 64, 32 or 16 half-word columns per CTA (even)
  const int cl = threadIdx.x % cols, slice = threadIdx.x / cols;
  const int h = blockIdx.x * cols + cl;  // half-word column: output columns 4 h .. 4 h + 3
  const int g = blockIdx.y;
  const int NW = N >> 3;
  const bool active = h < 2 * NW;  // both halves of a word are active together (N % 8 == 0)
  const int k0 = g * G + slice * kPackRows;
  float4 v[kPackRows];
  float mn[4] = {INFINITY, INFINITY, INFINITY, INFINITY}, mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  if (active) {
#pragma unroll
    for (int r = 0; r < kPackRows; ++r) v[r] = __ldg(reinterpret_cast<const float4*>(w + (size_t)(k0 + r) * N) + h);
#pragma unroll
    for (int r = 0; r < kPackRows; ++r) {
      mn[0] = fminf(mn[0], v[r].x), mx[0] = fmaxf(mx[0], v[r].x);
      mn[1] = fminf(mn[1], v[r].y), mx[1] = fmaxf(mx[1], v[r].y);
      mn[2] = fminf(mn[2], v[r].z), mx[2] = fmaxf(mx[2], v[r].z);
      mn[3] = fminf(mn[3], v[r].w), mx[3] = fmaxf(mx[3], v[r].w);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    red_mn[e][threadIdx.x] = mn[e];
    red_mx[e][threadIdx.x] = mx[e];
  }
  __syncthreads();
  // lanes beyond the last column leave; both lanes of a word are active together (N % 8 == 0), so
  // the shuffles below only ever pair active lanes
  const unsigned live = __ballot_sync(0xffffffffu, active);
  if (!active) return;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    for (int sl = 0; sl < slices; ++sl) {
      mn[e] = fminf(mn[e], red_mn[e][sl * cols + cl]);
      mx[e] = fmaxf(mx[e], red_mx[e][sl * cols + cl]);
    }
  }
  float s[4], inv[4], zf[4];
  uint32_t zhalf = 0u;
  __align__(8) __half sh[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __half hs = __float2half_rn(__fdiv_rn(__fsub_rn(mx[e], mn[e]), 15.0f));
    if ((__half_as_ushort(hs) & 0x7fffu) == 0) hs = __ushort_as_half(0x3c00u);
    sh[e] = hs;
    s[e] = __half2float(hs);
    inv[e] = __frcp_rn(s[e]);
    zf[e] = clamp_rint(__fdiv_rn(-mn[e], s[e]), 0.f, 15.f);
    zhalf |= (uint32_t)zf[e] << (4 * e);
  }
  const bool upper = h & 1;  // the upper half of its word: output columns 8 c + 4 .. 8 c + 7
  const int c = h >> 1;
  const uint32_t zother = __shfl_xor_sync(live, zhalf, 1);
  if (slice == 0) {
    *reinterpret_cast<uint2*>(scales + (size_t)g * N + 4 * h) = *reinterpret_cast<const uint2*>(sh);
    if (!upper) qzeros[(size_t)g * NW + c] = zhalf | (zother << 16);
  }
  // Codes through the product with 1 / s; a row with an element whose product lies within 2e-5 of
  // a rounding tie (rare) is redone with rint_div, which divides in that case.  Both give
  // round(v / s) exactly wherever they are used; r and z are integers, so r + z is exact.
#pragma unroll
  for (int r = 0; r < kPackRows; ++r) {
    const float e4[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
    uint32_t half = 0u;
    bool exact = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float t = __fmul_rn(e4[e], inv[e]);
      const float rt = rintf(t);
      exact |= fabsf(__fsub_rn(t, rt)) > 0.49998f;
      half |= (uint32_t)fminf(fmaxf(__fadd_rn(rt, zf[e]), 0.f), 15.f) << (4 * e);
    }
    if (exact) {
      half = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // codes saturate at 0 and 15 and z is in [0, 15]: |v / s| >= 64 clamps either way
        const float q = clamp_rint(__fadd_rn(rint_div(e4[e], s[e], inv[e], 64.f, 2e-5f), zf[e]), 0.f, 15.f);
        half |= (uint32_t)q << (4 * e);
      }
    }
    const uint32_t other = __shfl_xor_sync(live, half, 1);
    if (!upper) qweight[(size_t)(k0 + r) * NW + c] = half | (other << 16);
  }
  // The GEMMs read packed weights before waiting for the preceding kernel (programmatic dependent
  // launch): make this thread's writes visible device-wide before it exits, and so before this
  // grid completes, which is when a GEMM launched right after it on the stream may start.
  __threadfence();
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

// Per output column n: max_k |w[k, n]|, as the bit pattern of a non-negative float (whose unsigned
// order is the float order) reduced with atomicMax into wbits, which starts at 0.  A thread covers
// 4 consecutive columns (one 16-byte load per row) and a slice of the rows, kColRows rows per batch.
constexpr int kColRows = 8;

__global__ void __launch_bounds__(64)
    colmax_kernel(const float* __restrict__ w, int K, int N, int rows_per_cta, unsigned* __restrict__ wbits) {
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;  // column group of 4
  if (4 * c4 >= N) return;
  const int k0 = blockIdx.y * rows_per_cta;
  const int k1 = min(K, k0 + rows_per_cta);
  float m[4] = {0.f, 0.f, 0.f, 0.f};
  int k = k0;
  for (; k + kColRows <= k1; k += kColRows) {
    float4 v[kColRows];
#pragma unroll
    for (int r = 0; r < kColRows; ++r) v[r] = __ldg(reinterpret_cast<const float4*>(w + (size_t)(k + r) * N) + c4);
#pragma unroll
    for (int r = 0; r < kColRows; ++r) {
      m[0] = fmaxf(m[0], fabsf(v[r].x));
      m[1] = fmaxf(m[1], fabsf(v[r].y));
      m[2] = fmaxf(m[2], fabsf(v[r].z));
      m[3] = fmaxf(m[3], fabsf(v[r].w));
    }
  }
  for (; k < k1; ++k) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(w + (size_t)k * N) + c4);
    m[0] = fmaxf(m[0], fabsf(v.x));
    m[1] = fmaxf(m[1], fabsf(v.y));
    m[2] = fmaxf(m[2], fabsf(v.z));
    m[3] = fmaxf(m[3], fabsf(v.w));
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) atomicMax(wbits + 4 * c4 + e, __float_as_uint(m[e]));
}

// ws_n = absmax_n / Q_MAX (127 for int8 codes, 448 for e4m3; 1.0 for an all-zero column), in place
// over the max bit patterns.
__global__ void __launch_bounds__(256) colmax_scale_kernel(float* __restrict__ ws, int N, float qmax) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const float a = ws[n];
  ws[n] = a == 0.f ? 1.0f : __fdiv_rn(a, qmax);
  __threadfence();  // visible before the grid completes (see awq_pack_kernel)
}

// qw[n, k] = clamp(rint(w[k, n] / ws_n), -127, 127) (FP8: the e4m3 code of w[k, n] / ws_n),
// transposed through a 64 x 64 shared tile:
// thread (ty, tx) reads rows 4 ty .. 4 ty + 3 of columns 4 tx .. 4 tx + 3 (four 16-byte loads) and
// stores, per column, its four consecutive codes as one 32-bit word; then each thread writes 16 k
// of one output row.  K is a multiple of 16 and N of 32, so no piece straddles an edge.
constexpr int kQT = 64;
constexpr int kQTStride = kQT + 4;  // bytes per tile row: 4-byte stores of a warp spread over banks

template <bool FP8>
__global__ void __launch_bounds__(256)
    quant_transpose_kernel(const float* __restrict__ w, const float* __restrict__ ws, int K, int N,
                           uint8_t* __restrict__ qw) {
  __shared__ __align__(16) uint8_t tile[kQT * kQTStride];  // tile[n][k]
  // rows from the last tile down: the column-max pass reads high k last, so those rows are the
  // likeliest to be still in L2
  const int n0 = blockIdx.x * kQT, k0 = (gridDim.y - 1 - blockIdx.y) * kQT;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int n = n0 + 4 * tx;
  float sc[4] = {1.f, 1.f, 1.f, 1.f};
  if (n < N) {
    const float4 s4 = *reinterpret_cast<const float4*>(ws + n);
    sc[0] = s4.x, sc[1] = s4.y, sc[2] = s4.z, sc[3] = s4.w;
  }
  const float inv[4] = {__frcp_rn(sc[0]), __frcp_rn(sc[1]), __frcp_rn(sc[2]), __frcp_rn(sc[3])};
  float4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int k = k0 + 4 * ty + i;
    v[i] = (k < K && n < N) ? __ldg(reinterpret_cast<const float4*>(w + (size_t)k * N + n)) : make_float4(0, 0, 0, 0);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t word = 0u;
    if constexpr (FP8) {
      const float e[4] = {c == 0 ? v[0].x : c == 1 ? v[0].y : c == 2 ? v[0].z : v[0].w,
                          c == 0 ? v[1].x : c == 1 ? v[1].y : c == 2 ? v[1].z : v[1].w,
                          c == 0 ? v[2].x : c == 1 ? v[2].y : c == 2 ? v[2].z : v[2].w,
                          c == 0 ? v[3].x : c == 1 ? v[3].y : c == 2 ? v[3].z : v[3].w};
      word = e4m3x4_div(e, sc[c], inv[c]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float e = c == 0 ? v[i].x : c == 1 ? v[i].y : c == 2 ? v[i].z : v[i].w;
        // |w / ws| <= 127 + rounding by construction of ws; 256 bounds every unclamped value
        const float r = fminf(fmaxf(rint_div(e, sc[c], inv[c], 256.f, 1e-4f), -127.f), 127.f);
        word |= ((uint32_t)(int)r & 0xFFu) << (8 * i);
      }
    }
    *reinterpret_cast<uint32_t*>(tile + (4 * tx + c) * kQTStride + 4 * ty) = word;
  }
  __syncthreads();
  const int row = threadIdx.x >> 2, part = threadIdx.x & 3;  // output row n0 + row, k 16 part .. + 16
  const int nn = n0 + row, kk = k0 + 16 * part;
  if (nn < N && kk < K) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(tile + row * kQTStride + 16 * part);
    *reinterpret_cast<uint4*>(qw + (size_t)nn * K + kk) = make_uint4(src[0], src[1], src[2], src[3]);
  }
  __threadfence();  // the decode GEMMs read qw before their dependency wait (see awq_pack_kernel)
}

}  // namespace

cudaError_t launch_awq_pack(const float* w, int K, int N, int group, uint32_t* qweight, uint16_t* scales,
                            uint32_t* qzeros, cudaStream_t s) {
  const int NW = N / 8;
  const int cols = kPackThreads / (group / kPackRows);  // half-word columns per CTA
  dim3 block(kPackThreads), grid((2 * NW + cols - 1) / cols, K / group);
  awq_pack_kernel<<<grid, block, 0, s>>>(w, N, group, qweight, reinterpret_cast<__half*>(scales), qzeros);
  return cudaGetLastError();
}

cudaError_t launch_smooth(const float* absmax, const uint16_t* gamma, const float* w, int K, int N, float* s_out,
                          uint16_t* gamma_out, float* w_out, cudaStream_t s) {
  smooth_kernel<<<K, 256, 0, s>>>(absmax, reinterpret_cast<const __half*>(gamma), w, N, s_out,
                                  reinterpret_cast<__half*>(gamma_out), w_out);
  return cudaGetLastError();
}

namespace {
template <bool FP8>
cudaError_t launch_per_channel(const float* w, int K, int N, uint8_t* qw, float* ws, cudaStream_t s) {
  // 1. column maxima: about sixteen CTAs of 64 threads per SM, each over a slice of the rows
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(float) * (size_t)N, s);
  if (e != cudaSuccess) return e;
  const int col_ctas = (N / 4 + 63) / 64;
  int ks = (16 * num_sms() + col_ctas - 1) / col_ctas;
  if (ks > K / kColRows) ks = K / kColRows > 0 ? K / kColRows : 1;
  const int rows_per_cta = (K + ks - 1) / ks;
  colmax_kernel<<<dim3(col_ctas, (K + rows_per_cta - 1) / rows_per_cta), 64, 0, s>>>(
      w, K, N, rows_per_cta, reinterpret_cast<unsigned*>(ws));
  colmax_scale_kernel<<<(N + 255) / 256, 256, 0, s>>>(ws, N, FP8 ? 448.0f : 127.0f);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // 2. codes, transposed to [N, K]
  quant_transpose_kernel<FP8><<<dim3((N + kQT - 1) / kQT, (K + kQT - 1) / kQT), 256, 0, s>>>(w, ws, K, N, qw);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_per_channel_quant_i8(const float* w, int K, int N, int8_t* qw, float* ws, cudaStream_t s) {
  return launch_per_channel<false>(w, K, N, reinterpret_cast<uint8_t*>(qw), ws, s);
}

cudaError_t launch_per_channel_quant_fp8(const float* w, int K, int N, uint8_t* qw, float* ws, cudaStream_t s) {
  return launch_per_channel<true>(w, K, N, qw, ws, s);
}

}  // namespace wql
