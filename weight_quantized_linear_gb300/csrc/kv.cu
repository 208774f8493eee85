// kv.cu -- KV-cache int8 quantisation in groups of 128 channels and its dequantisation ("FastLLM
// architecture" article, section 5.2: the K and V cache kept in int8 with group size 128, turned
// back into fp16 when attention reads it).  A group is 128 consecutive channels of one row (one
// token's K or V vector); s = absmax / 127 in fp32 (1.0 for an all-zero group),
// q = clamp(rint(x / s), -128, 127), and the dequantised entry is fp16(q * s).
//
// Both kernels are streams over HBM: a half-warp owns a group (each lane 8 channels, one 16-byte
// load), the group's absmax is a 4-step shuffle within the half-warp, and each lane writes its 8
// codes as one 8-byte store (the half-warp's 128 codes are contiguous).  Persistent grid-stride
// warps; each iteration a warp takes kKvGroupsPerHalf groups per half-warp, all loaded before any
// is quantised, so that every thread keeps that many 16-byte loads in flight (2 -> 4 groups on
// 16384 x 8192 fp16: 95 -> 91 us).
#include "common.cuh"
#include "internal.h"

namespace wql {
namespace {

constexpr int kKvThreads = 256;
constexpr int kKvGroupsPerHalf = 4;  // groups per half-warp per iteration

// Eight fp16 (one uint4) widened to fp32.
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __low2float(h[i]);
    f[2 * i + 1] = __high2float(h[i]);
  }
}

// Low bytes of four ints, packed little-endian.
__device__ __forceinline__ uint32_t pack4(int c0, int c1, int c2, int c3) {
  return (uint32_t)(c0 & 0xff) | ((uint32_t)(c1 & 0xff) << 8) | ((uint32_t)(c2 & 0xff) << 16) |
         ((uint32_t)(c3 & 0xff) << 24);
}

// This lane's 8 channels of a group (channels 8 * sub .. + 7), whose other 120 channels are held by
// the other lanes of the half-warp.  Called by the whole warp at once (full-mask shuffles); a lane
// whose group is out of range computes on zeros and stores nothing.
__device__ __forceinline__ void quant_part(const uint4& raw, bool valid, long long g, int sub, int8_t* __restrict__ q,
                                           float* __restrict__ scales) {
  float x[8];
  unpack8(raw, x);
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = amax == 0.f ? 1.0f : __fdiv_rn(amax, 127.0f);
  const float inv = __fdiv_rn(1.0f, s);
  int c[8];
  bool exact = false;
#pragma unroll
  for (int e = 0; e < 8; ++e) c[e] = quant_fast(x[e], inv, exact);
  if (exact) {  // rare: a quotient within 5e-5 of a rounding tie
#pragma unroll
    for (int e = 0; e < 8; ++e) c[e] = quant_exact(x[e], s, inv);
  }
  if (!valid) return;
  __stcs(reinterpret_cast<uint2*>(q + g * 128 + 8 * sub),
         make_uint2(pack4(c[0], c[1], c[2], c[3]), pack4(c[4], c[5], c[6], c[7])));
  if (sub == 0) scales[g] = s;
}

// Groups are contiguous: group g covers kv elements [128 g, 128 g + 128).  With P =
// kKvGroupsPerHalf, warp w takes groups 2P w .. 2P w + 2P - 1, then 2P (w + W) .., half-warp h holding
// groups base + h + 2t (t < P).
__global__ void __launch_bounds__(kKvThreads) kv_quant_i8_kernel(const __half* __restrict__ kv, long long ngroups,
                                                                 int8_t* __restrict__ q, float* __restrict__ scales) {
  constexpr int P = kKvGroupsPerHalf;
  const int lane = threadIdx.x & 31, sub = lane & 15, h = lane >> 4;
  const long long warp = ((long long)blockIdx.x * kKvThreads + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * kKvThreads) >> 5;
  const uint4* src = reinterpret_cast<const uint4*>(kv);
  for (long long base = 2 * P * warp; base < ngroups; base += 2 * P * nwarps) {  // uniform over the warp
    uint4 raw[P];
#pragma unroll
    for (int t = 0; t < P; ++t) {
      const long long g = base + h + 2 * t;
      raw[t] = g < ngroups ? __ldcs(src + g * 16 + sub) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int t = 0; t < P; ++t) {
      const long long g = base + h + 2 * t;
      quant_part(raw[t], g < ngroups, g, sub, q, scales);
    }
  }
}

// out = fp16(q * s) (the fp32 product rounded once more, to fp16).  A lane dequantises 8 channels:
// one 8-byte load of codes, one 16-byte store.
__global__ void __launch_bounds__(kKvThreads) kv_dequant_i8_kernel(const int8_t* __restrict__ q,
                                                                   const float* __restrict__ scales, long long n8,
                                                                   __half* __restrict__ out) {
  const long long stride = (long long)gridDim.x * kKvThreads;
  for (long long i = (long long)blockIdx.x * kKvThreads + threadIdx.x; i < n8; i += stride) {
    const uint2 c = __ldcs(reinterpret_cast<const uint2*>(q) + i);
    const float s = __ldg(scales + (i >> 4));  // 16 lanes of 8 channels per group
    const uint32_t w[2] = {c.x, c.y};
    __align__(16) __half2 o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int b0 = (int)(int8_t)(w[j >> 1] >> (16 * (j & 1))), b1 = (int)(int8_t)(w[j >> 1] >> (16 * (j & 1) + 8));
      o[j] = __halves2half2(__float2half_rn(__fmul_rn(__int2float_rn(b0), s)),
                            __float2half_rn(__fmul_rn(__int2float_rn(b1), s)));
    }
    __stcs(reinterpret_cast<uint4*>(out) + i, *reinterpret_cast<const uint4*>(o));
  }
}

int kv_grid(long long units_per_cta, long long units) {
  const long long want = (units + units_per_cta - 1) / units_per_cta;
  const long long cap = 8LL * num_sms();  // eight CTAs of 256 threads per SM
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_kv_quant_i8(const uint16_t* kv, long long rows, int D, int8_t* q, float* scales, cudaStream_t s) {
  const long long ngroups = rows * (D / 128);
  if (ngroups == 0) return cudaSuccess;
  kv_quant_i8_kernel<<<kv_grid(kKvThreads / 16 * kKvGroupsPerHalf, ngroups), kKvThreads, 0, s>>>(
      reinterpret_cast<const __half*>(kv), ngroups, q, scales);
  return cudaGetLastError();
}

cudaError_t launch_kv_dequant_i8(const int8_t* q, const float* scales, long long rows, int D, uint16_t* out,
                                 cudaStream_t s) {
  const long long n8 = rows * (long long)D / 8;
  if (n8 == 0) return cudaSuccess;
  kv_dequant_i8_kernel<<<kv_grid(kKvThreads, n8), kKvThreads, 0, s>>>(q, scales, n8, reinterpret_cast<__half*>(out));
  return cudaGetLastError();
}

}  // namespace wql
