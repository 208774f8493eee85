// w8a8_decode.cu -- SmoothQuant W8A8 GEMM for decode-shaped calls ("LMDeploy W8A8 quantisation
// guide", QLinear.forward / matmul_kernel_dynamic_quant: int8 x int8 products accumulated in
// int32, then c = c * rms_scale * linear_scale in fp32 and rounded to fp16).
//
// GB300 has no int8 path in tcgen05 and its legacy int8 mma.sync runs at a quarter of the fp16
// rate, so int8 values are converted exactly to fp16 in registers (PRMT places each biased byte in
// the mantissa of 1024 + b + 128, one f16x2 add removes 1152) and multiplied on the fp16
// mma.sync.m16n8k16 path with fp32 accumulation.  Products are at most 128 * 127 = 16256 < 2^14;
// each thread folds its fp32 partial sums into int32 before they can cover more than 1024
// products (< 2^24), so every partial sum is an integer that fp32 holds exactly and the int32
// result is exact for every input.
//
// Weights are the 16-row MMA operand ("swap AB"), tokens the 8-column operand.  Weight tiles of
// 128 output channels x 64 k stream once from HBM through a TMA pipeline; split-K across the
// CTAs of a cluster, reduced through distributed shared memory in int32.
//
// The fp8 variant (the page's quant_dtype fp8, float8_e4m3fn codes, fp32 accumulator) runs the same
// pipeline: every e4m3 value is an fp16 value, so one cvt per pair of codes feeds the same fp16
// MMA; its fp32 sums are not folded, and the split-K partials are added in fp32 in rank order.
#include <atomic>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace wql {
namespace {

constexpr int kBK = 64;            // k per stage (bytes of a weight row)
constexpr int kRows = 128;         // output channels per CTA
constexpr int kConsumerWarps = 8;  // 4 tile pairs x 2 k16 phases
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxCluster = 8;
constexpr int kFoldStages = 32;    // each warp sees 32 k per stage: fold to int32 every 1024 k

template <int MT>
struct Layout8 {
  static constexpr int kXBytes = 8 * MT * kBK;  // token rows x 64 B
  static constexpr int kWBytes = kRows * kBK;   // 128 rows x 64 B
  static constexpr int kStage = (kXBytes + kWBytes + 1023) / 1024 * 1024;
  static constexpr int kStages = 8;
  static constexpr int kPipe = kStages * kStage;
  static constexpr int kRed = 2 * 8 * MT * kRows * 4;  // [2 k phases][tokens][128] int32
  static constexpr int kData = kPipe > kRed ? kPipe : kRed;
  static constexpr int kRecv = (8 * MT * kRows / 4 + kMaxCluster) * 16;  // owner's receive slots, dedicated
  static constexpr int kBytes = kData + kRecv + 1024 + 2 * kStages * 8;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Byte offset of 4-byte word t of 16-byte chunk c in row r of a 64-byte-row tile, 64B swizzle.
__device__ __forceinline__ uint32_t tile64_off(int r, int c, int t) {
  return r * 64 + (((c ^ (r >> 1)) & 3) << 4) + t * 4;
}

// Four 8-bit codes -> two f16x2 (bytes 0,1 and bytes 2,3), exact.  int8: each biased byte is placed
// in the mantissa of 1024 + b + 128 and one f16x2 add removes 1152; e4m3: the hardware conversion.
template <bool FP8>
__device__ __forceinline__ void q8x4_to_h2x2(uint32_t v, uint32_t& lo, uint32_t& hi) {
  if constexpr (FP8) {
    e4m3x4_to_f16x2x2(v, lo, hi);
  } else {
    const uint32_t u = v ^ 0x80808080u;
    lo = hadd2_u32(prmt(u, 0x64646464u, 0x4140u), 0xE480E480u);
    hi = hadd2_u32(prmt(u, 0x64646464u, 0x4342u), 0xE480E480u);
  }
}

template <int MT, bool FP8>
__global__ void __launch_bounds__(kThreads, MT <= 2 ? 2 : 1)
    w8a8_decode_kernel(const __grid_constant__ CUtensorMap tm_x,  // q [M][K] 8-bit codes, box {64, 8MT}, SW64
                       const __grid_constant__ CUtensorMap tm_w,  // qw [N][K] 8-bit codes, box {64, 128}, SW64
                       const float* __restrict__ xs, const float* __restrict__ ws, int M, int N, int kblocks,
                       __half* y, void* __restrict__ acc_out, EpilogueAdd ea, unsigned* err) {
  using L = Layout8<MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  int4* recv = reinterpret_cast<int4*>(smem + L::kData);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kData + L::kRecv);
  uint64_t* empty = full + L::kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int strip = blockIdx.x;
  const int split = blockIdx.y, nsplit = gridDim.y;
  const int m0 = blockIdx.z * 8 * MT;
  const int kb0 = (int)((long long)kblocks * split / nsplit);
  const int kb1 = (int)((long long)kblocks * (split + 1) / nsplit);

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbarrier_init();
  }
  __syncwarp();
  cluster_arrive_relaxed();  // matched by cluster_wait() before the first remote store
  __syncthreads();

  const int g = lane >> 2, t = lane & 3;
  const int tp = warp & 3, kp = warp >> 2;  // tile pair (32 channels) and k16 phase
  int tot[2][MT][4];  // int8: exact int32 sums; fp8: the bits of the fp32 sums
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) tot[a][mt][i] = 0;

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_w);
      const uint64_t pol = policy_evict_first();
      const uint32_t bytes = L::kXBytes + L::kWBytes;
      const int nkb = kb1 - kb0;
      // prologue: weight tiles first (independent of the previous kernel), activations after the
      // programmatic dependency resolves
      const int pro = nkb < L::kStages ? nkb : L::kStages;
      for (int i = 0; i < pro; ++i) {
        mbar_arrive_expect_tx(&full[i], bytes);
        tma_load_2d_hint(smem + i * L::kStage + L::kXBytes, &tm_w, &full[i], (kb0 + i) * kBK, strip * kRows, pol);
      }
      grid_dependency_wait();
      for (int i = 0; i < pro; ++i) tma_load_2d(smem + i * L::kStage, &tm_x, &full[i], (kb0 + i) * kBK, m0);
      // the next kernel may launch now: its CTAs open with a burst of weight copies on these SMs'
      // TMA units, which must not queue ahead of the activation copies above
      grid_dependents_launch();
      int issued = pro;
      for (; issued < nkb; ++issued) {
        const int s = issued % L::kStages;
        const int kb = kb0 + issued;
        if (!mbar_wait_bounded(&empty[s], ((issued / L::kStages) & 1) ^ 1)) {
          report_error(err, kErrTimeoutEmpty);
          break;
        }
        uint8_t* st = smem + s * L::kStage;
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_2d_hint(st + L::kXBytes, &tm_w, &full[s], kb * kBK, strip * kRows, pol);
        tma_load_2d(st, &tm_x, &full[s], kb * kBK, m0);
      }
      const int n = issued < L::kStages ? issued : L::kStages;
      for (int i = issued - n; i < issued; ++i) {
        if (!mbar_wait_bounded(&full[i % L::kStages], (i / L::kStages) & 1)) {
          report_error(err, kErrTimeoutDrain);
          break;
        }
      }
    }
  } else {
    float acc[2][MT][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[a][mt][i] = 0.f;

    auto fold = [&]() {
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if constexpr (FP8) {
              tot[a][mt][i] = __float_as_int(acc[a][mt][i]);
            } else {
              tot[a][mt][i] += __float2int_rn(acc[a][mt][i]);
              acc[a][mt][i] = 0.f;
            }
          }
    };

    int it = 0;
    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const int s = it % L::kStages;
      if (!mbar_wait_bounded(&full[s], (it / L::kStages) & 1)) {
        report_error(err, kErrTimeoutFull);
        break;
      }
      const uint32_t xt = smem_u32(smem + s * L::kStage);
      const uint32_t wt = xt + L::kXBytes;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = kp + 2 * h;  // 16-byte chunk = k16 step within the stage
        uint32_t bx[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          q8x4_to_h2x2<FP8>(lds_u32(xt + tile64_off(8 * mt + g, c, t)), bx[mt][0], bx[mt][1]);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          const int r = 32 * tp + 16 * a + g;
          uint32_t A[4];
          q8x4_to_h2x2<FP8>(lds_u32(wt + tile64_off(r, c, t)), A[0], A[2]);
          q8x4_to_h2x2<FP8>(lds_u32(wt + tile64_off(r + 8, c, t)), A[1], A[3]);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) mma_f16_16816(acc[a][mt], A, bx[mt][0], bx[mt][1]);
        }
      }
      // generic-proxy reads of the stage are ordered before its TMA refill (async proxy) only by
      // a proxy fence; the mbarrier release alone does not do it
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (!FP8 && (it + 1) % kFoldStages == 0) fold();
    }
    fold();
  }

  __syncthreads();
  int* red = reinterpret_cast<int*>(smem);
  constexpr int kE = 8 * MT * kRows;
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = 8 * mt + 2 * t + (i & 1);
          const int col = 32 * tp + 16 * a + g + 8 * (i >> 1);
          red[kp * kE + row * kRows + col] = tot[a][mt][i];
        }
  }
  __syncthreads();
  __syncwarp();
  cluster_wait();  // every peer has started: its receive buffer may be written
  const uint32_t rank = cluster_ctarank();
  const int nq = kE / 4;
  const int lmax = (nq + nsplit - 1) / nsplit;
  // int4 of int32 sums, or of fp32 bit patterns
  auto add4 = [](int4 a, int4 b) {
    if constexpr (FP8)
      return make_int4(__float_as_int(__fadd_rn(__int_as_float(a.x), __int_as_float(b.x))),
                       __float_as_int(__fadd_rn(__int_as_float(a.y), __int_as_float(b.y))),
                       __float_as_int(__fadd_rn(__int_as_float(a.z), __int_as_float(b.z))),
                       __float_as_int(__fadd_rn(__int_as_float(a.w), __int_as_float(b.w))));
    else
      return make_int4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
  };
  {  // fold the two k-phase partials and push each slice to its owner
    const int4* r4 = reinterpret_cast<const int4*>(red);
    for (int f = threadIdx.x; f < nq; f += kThreads) {
      const int owner = slice_owner(f, nq, nsplit);
      const int f0 = (int)((long long)nq * owner / nsplit);
      st_cluster_i4(map_cluster(recv + rank * lmax + (f - f0), owner), add4(r4[f], r4[nq + f]));
    }
  }
  __syncwarp();
  cluster_sync();  // all slices delivered
  {
    const int f0 = (int)((long long)nq * rank / nsplit), f1 = (int)((long long)nq * (rank + 1) / nsplit);
    for (int f = f0 + threadIdx.x; f < f1; f += kThreads) {
      int4 v = recv[f - f0];
      for (int q = 1; q < nsplit; ++q) v = add4(v, recv[q * lmax + (f - f0)]);
      const int row = (4 * f) / kRows, col = (4 * f) % kRows;
      const int m = m0 + row, n = strip * kRows + col;
      if (m < M && n < N) {
        const float xm = xs[m];
        const float4 wn = *reinterpret_cast<const float4*>(ws + n);
        const int iv[4] = {v.x, v.y, v.z, v.w};
        const float wv[4] = {wn.x, wn.y, wn.z, wn.w};
        float bv[4] = {0.f, 0.f, 0.f, 0.f}, rv[4] = {0.f, 0.f, 0.f, 0.f};
        if (ea.bias) load_half4(ea.bias + n, bv);
        if (ea.residual) load_half4(ea.residual + (size_t)m * N + n, rv);
        __align__(8) __half hv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float c = FP8 ? __int_as_float(iv[e]) : __int2float_rn(iv[e]);
          hv[e] = __float2half_rn(add_terms(__fmul_rn(__fmul_rn(c, xm), wv[e]), ea, bv[e], rv[e]));
        }
        *reinterpret_cast<uint2*>(y + (size_t)m * N + n) = *reinterpret_cast<const uint2*>(hv);
        if (acc_out) reinterpret_cast<int4*>(acc_out)[((size_t)m * N + n) / 4] = v;
      }
    }
  }
}

template <int MT, bool FP8>
cudaError_t launch8(const CUtensorMap& tx, const CUtensorMap& tw, const float* xs, const float* ws, int M, int N,
                    int kblocks, __half* y, void* acc_out, EpilogueAdd ea, unsigned* dev_err, cudaStream_t stream) {
  using L = Layout8<MT>;
  // 8- and 16-token launches take the same shared-memory footprint, so that back-to-back layers
  // look alike to the block scheduler whatever their token counts: it then keeps one CTA of each
  // of two consecutive layers per SM (M = 1 then M = 16 layers at N = 4096: 8.17 -> 6.88 us per
  // launch; with unequal footprints some SMs held two CTAs of one layer)
  const int bytes = MT <= 2 ? (Layout8<1>::kBytes > Layout8<2>::kBytes ? Layout8<1>::kBytes : Layout8<2>::kBytes)
                            : L::kBytes;
  static std::atomic<bool> attr_set[64];  // per device; racing first calls set the same attribute
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(w8a8_decode_kernel<MT, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const int strips = (N + kRows - 1) / kRows;
  const int mblocks = (M + 8 * MT - 1) / (8 * MT);
  const int S = pick_k_split(reinterpret_cast<const void*>(w8a8_decode_kernel<MT, FP8>), kThreads, bytes, strips * mblocks,
                             kblocks, /*pow2=*/false, /*balanced=*/true);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(strips, S, mblocks);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 1;
  attrs[0].val.clusterDim.y = S;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, w8a8_decode_kernel<MT, FP8>, tx, tw, xs, ws, M, N, kblocks, y, acc_out, ea, dev_err);
}

template <bool FP8>
cudaError_t launch_decode(const void* q, const float* xs, const void* qw, const float* ws, int M, int K, int N,
                          uint16_t* y, void* acc_out, const uint16_t* bias, const uint16_t* residual, unsigned* dev_err,
                          cudaStream_t stream, std::string* err) {
  const int MT = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
  const EpilogueAdd ea{reinterpret_cast<const __half*>(bias), reinterpret_cast<const __half*>(residual)};
  CUtensorMap tx, tw;
  if (!make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q, K, M, (uint64_t)K, kBK, 8 * MT,
                    CU_TENSOR_MAP_SWIZZLE_64B, err) ||
      !make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qw, K, N, (uint64_t)K, kBK, kRows,
                    CU_TENSOR_MAP_SWIZZLE_64B, err)) {
    return cudaErrorInvalidValue;
  }
  const int kblocks = (K + kBK - 1) / kBK;
  __half* yh = reinterpret_cast<__half*>(y);
  switch (MT) {
    case 1:
      return launch8<1, FP8>(tx, tw, xs, ws, M, N, kblocks, yh, acc_out, ea, dev_err, stream);
    case 2:
      return launch8<2, FP8>(tx, tw, xs, ws, M, N, kblocks, yh, acc_out, ea, dev_err, stream);
    default:
      return launch8<4, FP8>(tx, tw, xs, ws, M, N, kblocks, yh, acc_out, ea, dev_err, stream);
  }
}

}  // namespace

cudaError_t launch_w8a8_decode(const int8_t* q, const float* xs, const int8_t* qw, const float* ws, int M, int K,
                               int N, uint16_t* y, int32_t* acc_out, const uint16_t* bias, const uint16_t* residual,
                               unsigned* dev_err, cudaStream_t stream, std::string* err) {
  return launch_decode<false>(q, xs, qw, ws, M, K, N, y, acc_out, bias, residual, dev_err, stream, err);
}

cudaError_t launch_fp8_decode(const uint8_t* q, const float* xs, const uint8_t* qw, const float* ws, int M, int K,
                              int N, uint16_t* y, float* acc_out, const uint16_t* bias, const uint16_t* residual,
                              unsigned* dev_err, cudaStream_t stream, std::string* err) {
  return launch_decode<true>(q, xs, qw, ws, M, K, N, y, acc_out, bias, residual, dev_err, stream, err);
}

}  // namespace wql
