// norm.cu -- QRMSNorm fused with per-token dynamic int8 or fp8 quantisation, the same per-token
// quantisation of a row without the norm, and the calibration statistic used by weight smoothing ("LMDeploy W8A8 quantisation guide": QRMSNorm.forward,
// rms_norm_dynamic_quant, per_token_quant_int8 with scale = absmax / Q_MAX; int8 codes are rounded
// to integers (Q_MAX = 127), fp8 codes are the e4m3 cast (Q_MAX = 448); smoothing statistics are
// the per-channel absmax of the norm output).
//
// CTAs of 256 threads walk the token rows; each row is brought into shared memory by a bulk copy
// (several rows in flight per CTA) and held in registers while it is normalised.  The sum of
// squares uses a fixed order (chunk c of 8 elements belongs to thread
// c mod 256, which adds its elements in increasing k; the 256 partial sums are then folded
// pairwise (t, t+128), (t, t+64), ..., (t, t+1)), so int8 codes are reproducible bit for bit.
// Every float operation uses an explicitly rounded intrinsic: nothing is contracted into FMA.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace wql {
namespace {

constexpr int kNormThreads = 256;

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

// Bulk copy of `bytes` contiguous bytes from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Modes of the row kernel: 0 int8 codes, 1 per-channel absmax (atomic max into absmax), 2 residual
// add then int8 codes, 3 fp8 codes, 4 residual add then fp8 codes, 5 int8 and 6 fp8 codes of the row
// itself (per_token_quant: no normalisation, no gamma).
__host__ __device__ constexpr bool mode_residual(int mode) { return mode == 2 || mode == 4; }
__host__ __device__ constexpr bool mode_fp8(int mode) { return mode == 3 || mode == 4 || mode == 6; }
__host__ __device__ constexpr bool mode_no_norm(int mode) { return mode == 5 || mode == 6; }

// Rows in flight per CTA: four, or three when each slot holds two long rows (residual, K > 8192).
__host__ __device__ constexpr int norm_slots(int cpt, int mode) { return (mode_residual(mode) && cpt > 4) ? 3 : 4; }
__host__ __device__ constexpr int norm_rows_per_slot(int mode) { return mode_residual(mode) ? 2 : 1; }

// Low bytes of four ints, packed little-endian.
__device__ __forceinline__ uint32_t pack_s8x4(int c0, int c1, int c2, int c3) {
  const uint32_t lo = prmt((uint32_t)c0, (uint32_t)c1, 0x0040u), hi = prmt((uint32_t)c2, (uint32_t)c3, 0x0040u);
  return prmt(lo, hi, 0x5410u);
}

// Sum of the 256 lane partials in the fixed order (t, t+128), (t, t+64), ..., (t, t+1), with one
// barrier: every warp evaluates the three cross-warp levels (lane l from the eight partials
// l + 32 w, in exactly that order) and the five shuffle levels itself, so all threads get the same
// total.  The barrier also votes: it returns false in every thread if `ok` is false in any thread.
__device__ __forceinline__ bool row_sum_vote(float p, bool ok, float* red, float& total) {
  const int lane = threadIdx.x & 31;
  red[threadIdx.x] = p;
  if (__syncthreads_or(!ok)) return false;
  const float* r = red + lane;
  const float a0 = __fadd_rn(r[0], r[128]), a1 = __fadd_rn(r[64], r[192]);
  const float a2 = __fadd_rn(r[32], r[160]), a3 = __fadd_rn(r[96], r[224]);
  const float b0 = __fadd_rn(a0, a1), b1 = __fadd_rn(a2, a3);
  float v = __fadd_rn(b0, b1);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
  total = __shfl_sync(0xffffffffu, v, 0);
  return true;
}

// Quantising modes write (q, xs); MODE 1 writes the per-channel absmax of the norm output.  The
// residual modes add the residual first ("LMDeploy W8A8 quantisation guide", inference kernels: the
// residual fusion of rms_norm_dynamic_quant): h = fp16(fp32(x) + fp32(r)) is stored to h_out (the
// new residual; it may be the residual buffer itself) and normalised and quantised like x.
// Persistent CTAs: CTA b normalises rows b, b + gridDim.x, ...  Thread 0 keeps kNormSlots rows in
// flight with bulk copies into a shared-memory ring, so HBM reads continue through every row's
// reductions; a slot is refilled as soon as all threads have read it (the first barrier of the
// row's sum).
template <int CPT, int MODE>
// (the residual mode holds the new residual across the row sum: three CTAs per SM, no spill)
__global__ void __launch_bounds__(kNormThreads, CPT <= 2 ? (mode_residual(MODE) ? 3 : 4) : 1)
    qrmsnorm_kernel(const __half* __restrict__ x, const __half* residual, const __half* __restrict__ gamma, float eps,
                    int M, int K, uint8_t* __restrict__ q, float* __restrict__ xs, float* __restrict__ absmax,
                    __half* h_out, unsigned* err) {
  constexpr int kNormSlots = norm_slots(CPT, MODE), kRowsPerSlot = norm_rows_per_slot(MODE);
  constexpr bool kResid = mode_residual(MODE);
  constexpr bool kNorm = !mode_no_norm(MODE);
  __shared__ float red[272];  // [0, 256) lane partials, 256 row sum, [264, 272) warp maxima
  __shared__ __align__(8) uint64_t full[kNormSlots];
  extern __shared__ __align__(16) uint8_t rows[];  // kNormSlots x kRowsPerSlot x 2K bytes
  const int tid = threadIdx.x;
  const int nchunks = K >> 3;
  const uint32_t row_bytes = 2u * (uint32_t)K;
  const uint32_t slot_bytes = kRowsPerSlot * row_bytes;
  const int nrows = M > (int)blockIdx.x ? (M - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  auto issue = [&](int j) {  // row j of this CTA (and its residual row) into slot j % kNormSlots
    const int s = j % kNormSlots;
    const size_t off = (size_t)(blockIdx.x + (size_t)j * gridDim.x) * K;
    mbar_arrive_expect_tx(&full[s], slot_bytes);
    bulk_load(rows + (size_t)s * slot_bytes, x + off, row_bytes, &full[s]);
    if constexpr (kResid) bulk_load(rows + (size_t)s * slot_bytes + row_bytes, residual + off, row_bytes, &full[s]);
  };
  if (tid == 0) {
    for (int s = 0; s < kNormSlots; ++s) mbar_init(&full[s], 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  // x comes from the preceding kernel, which may also still read q and xs
  grid_dependency_wait();
  if (tid == 0) {
    for (int j = 0; j < nrows && j < kNormSlots; ++j) issue(j);
    grid_dependents_launch();  // the next kernel's copies now queue behind these
  }
  // gamma is read once per CTA and kept in registers, as fp32, for all of its rows
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  float gf[CPT][8];
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int c = tid + kNormThreads * i;
    if (kNorm && c < nchunks) {
      const uint4 gv = __ldg(gr + c);
      const __half* gh = reinterpret_cast<const __half*>(&gv);
#pragma unroll
      for (int e = 0; e < 8; ++e) gf[i][e] = __half2float(gh[e]);
    }
  }

  int j = 0;
  for (; j < nrows; ++j) {
    const int m = blockIdx.x + j * gridDim.x;
    const int s = j % kNormSlots;
    // Every thread waits; the row sum's barrier votes, so that all threads leave together if a wait
    // ever expires (the values read from an unfinished slot are then discarded).
    const bool ok = mbar_wait_bounded(&full[s], (j / kNormSlots) & 1);
    const uint4* xr = reinterpret_cast<const uint4*>(rows + (size_t)s * slot_bytes);
    float yv[CPT][8];  // x (or x + r as fp16), then the normalised row
    uint4 hv[kResid ? CPT : 1];  // the new residual, stored once the row's wait is confirmed
    float p = 0.f;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = tid + kNormThreads * i;
      if (c < nchunks) {
        uint4 xv = xr[c];
        if constexpr (kResid) {
          const uint4 rv = reinterpret_cast<const uint4*>(rows + (size_t)s * slot_bytes + row_bytes)[c];
          const __half* xh = reinterpret_cast<const __half*>(&xv);
          const __half* rh = reinterpret_cast<const __half*>(&rv);
          __align__(16) __half hh[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) hh[e] = __float2half_rn(__fadd_rn(__half2float(xh[e]), __half2float(rh[e])));
          hv[i] = *reinterpret_cast<const uint4*>(hh);
          xv = hv[i];
        }
        const __half* h = reinterpret_cast<const __half*>(&xv);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float v = __half2float(h[e]);
          yv[i][e] = v;
          if constexpr (kNorm) p = __fadd_rn(p, __fmul_rn(v, v));
        }
      }
    }
    // the slot was read through the generic proxy and thread 0 refills it with a bulk copy (async
    // proxy) after the next barrier: a proxy fence orders the reads before that write
    fence_proxy_async_smem();
    float ss;
    if (!row_sum_vote(p, ok, red, ss)) {
      if (tid == 0) report_error(err, kErrTimeoutFull);
      break;
    }
    // every thread has read slot s (it passed the sum's barrier): refill it
    if (tid == 0 && j + kNormSlots < nrows) issue(j + kNormSlots);
    if constexpr (kResid) {
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = tid + kNormThreads * i;
        if (c < nchunks) *reinterpret_cast<uint4*>(h_out + (size_t)m * K + 8 * c) = hv[i];
      }
    }
    float amax = 0.f;
    if constexpr (kNorm) {
      const float mean = __fdiv_rn(ss, (float)K);
      const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = tid + kNormThreads * i;
        if (c < nchunks) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float yy = __fmul_rn(__fmul_rn(yv[i][e], r), gf[i][e]);
            yv[i][e] = yy;
            amax = fmaxf(amax, fabsf(yy));
          }
        }
      }
    } else {  // per-token quantisation of the row itself
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = tid + kNormThreads * i;
        if (c < nchunks) {
#pragma unroll
          for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(yv[i][e]));
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
      __syncthreads();  // the lane partials in red[] are read by every warp before the next row writes them
      continue;
    }

    const float rowmax = block_max(amax, red);
    const float scale = rowmax == 0.f ? 1.0f : __fdiv_rn(rowmax, mode_fp8(MODE) ? 448.0f : 127.0f);
    const float inv = __fdiv_rn(1.0f, scale);
    if (tid == 0) xs[m] = scale;
    uint8_t* qr = q + (size_t)m * K;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = tid + kNormThreads * i;
      if (mode_fp8(MODE) && c < nchunks) {
        const float y0[4] = {yv[i][0], yv[i][1], yv[i][2], yv[i][3]};
        const float y1[4] = {yv[i][4], yv[i][5], yv[i][6], yv[i][7]};
        *reinterpret_cast<uint2*>(qr + 8 * c) = make_uint2(e4m3x4_div(y0, scale, inv), e4m3x4_div(y1, scale, inv));
      } else if (c < nchunks) {
        int k8[8];
        bool exact = false;
#pragma unroll
        for (int e = 0; e < 8; ++e) k8[e] = quant_fast(yv[i][e], inv, exact);
        if (exact) {  // rare: some element lies within 5e-5 of a rounding tie
#pragma unroll
          for (int e = 0; e < 8; ++e) k8[e] = quant_exact(yv[i][e], scale, inv);
        }
        *reinterpret_cast<uint2*>(qr + 8 * c) =
            make_uint2(pack_s8x4(k8[0], k8[1], k8[2], k8[3]), pack_s8x4(k8[4], k8[5], k8[6], k8[7]));
      }
    }
  }
  // Leave no copy in flight: after an expired wait, wait (bounded) for the rows still issued.
  if (j < nrows && tid == 0) {
    const int issued = nrows < j + kNormSlots ? nrows : j + kNormSlots;
    for (int i = j; i < issued; ++i)
      if (!mbar_wait_bounded(&full[i % kNormSlots], (i / kNormSlots) & 1)) {
        report_error(err, kErrTimeoutDrain);
        break;
      }
  }
}

// Launch with programmatic stream serialisation: the kernel may start while its predecessor drains
// (it waits with griddepcontrol.wait before touching its inputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

template <int CPT, int MODE>
cudaError_t launch_rows(const __half* x, const __half* residual, const __half* gamma, float eps, int M, int K,
                        uint8_t* q, float* xs, float* absmax, __half* h_out, unsigned* err, cudaStream_t s) {
  auto kern = qrmsnorm_kernel<CPT, MODE>;
  const size_t smem = (size_t)norm_slots(CPT, MODE) * norm_rows_per_slot(MODE) * 2 * K;
  // Per device: the dynamic shared-memory limit set on this kernel, and the occupancy of the ring
  // size last asked for.  They change together and only when a row length needs a larger ring, so
  // one mutex keeps them consistent across host threads (an uncontended lock per call).
  static std::mutex mu;
  static int set_bytes[64] = {0};
  static int fit_bytes[64] = {0};
  static int fit_ctas[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) return cudaErrorInvalidDevice;
  int ctas = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (set_bytes[dev] < (int)smem) {  // a longer row needs a larger ring: raise the limit
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      set_bytes[dev] = (int)smem;
    }
    if (fit_bytes[dev] != (int)smem) {
      int fit = 0;
      cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, kern, kNormThreads, smem);
      if (e != cudaSuccess) return e;
      fit_bytes[dev] = (int)smem;
      fit_ctas[dev] = fit > 0 ? fit : 1;
    }
    ctas = fit_ctas[dev];
  }
  const long long cap = (long long)ctas * num_sms();
  const dim3 grid((unsigned)(M < cap ? M : cap)), block(kNormThreads);
  return launch_pdl(kern, grid, block, smem, s, x, residual, gamma, eps, M, K, q, xs, absmax, h_out, err);
}

template <int MODE>
cudaError_t launch_norm(const uint16_t* x, const uint16_t* residual, const uint16_t* gamma, float eps, int M, int K,
                        uint8_t* q, float* xs, float* absmax, uint16_t* h_out, unsigned* err, cudaStream_t s) {
  const __half* xh = reinterpret_cast<const __half*>(x);
  const __half* rh = reinterpret_cast<const __half*>(residual);
  const __half* gh = reinterpret_cast<const __half*>(gamma);
  __half* hh = reinterpret_cast<__half*>(h_out);
  const int cpt = (K + 2047) / 2048;
  if (cpt <= 1) return launch_rows<1, MODE>(xh, rh, gh, eps, M, K, q, xs, absmax, hh, err, s);
  if (cpt <= 2) return launch_rows<2, MODE>(xh, rh, gh, eps, M, K, q, xs, absmax, hh, err, s);
  if (cpt <= 4) return launch_rows<4, MODE>(xh, rh, gh, eps, M, K, q, xs, absmax, hh, err, s);
  return launch_rows<8, MODE>(xh, rh, gh, eps, M, K, q, xs, absmax, hh, err, s);
}

}  // namespace

cudaError_t launch_qrmsnorm_quant_i8(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K, int8_t* q,
                                     float* xs, unsigned* dev_err, cudaStream_t s) {
  return launch_norm<0>(x, nullptr, gamma, eps, M, K, reinterpret_cast<uint8_t*>(q), xs, nullptr, nullptr, dev_err, s);
}

cudaError_t launch_add_qrmsnorm_quant_i8(const uint16_t* x, const uint16_t* residual, const uint16_t* gamma,
                                         float eps, int M, int K, uint16_t* residual_out, int8_t* q, float* xs,
                                         unsigned* dev_err, cudaStream_t s) {
  return launch_norm<2>(x, residual, gamma, eps, M, K, reinterpret_cast<uint8_t*>(q), xs, nullptr, residual_out,
                        dev_err, s);
}

cudaError_t launch_qrmsnorm_quant_fp8(const uint16_t* x, const uint16_t* residual, const uint16_t* gamma, float eps,
                                      int M, int K, uint16_t* residual_out, uint8_t* q, float* xs, unsigned* dev_err,
                                      cudaStream_t s) {
  if (residual) return launch_norm<4>(x, residual, gamma, eps, M, K, q, xs, nullptr, residual_out, dev_err, s);
  return launch_norm<3>(x, nullptr, gamma, eps, M, K, q, xs, nullptr, nullptr, dev_err, s);
}

cudaError_t launch_per_token_quant(const uint16_t* x, int M, int K, bool fp8, uint8_t* q, float* xs, unsigned* dev_err,
                                   cudaStream_t s) {
  if (fp8) return launch_norm<6>(x, nullptr, nullptr, 0.f, M, K, q, xs, nullptr, nullptr, dev_err, s);
  return launch_norm<5>(x, nullptr, nullptr, 0.f, M, K, q, xs, nullptr, nullptr, dev_err, s);
}

cudaError_t launch_act_absmax(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K, float* absmax,
                              unsigned* dev_err, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(absmax, 0, sizeof(float) * (size_t)K, s);
  if (e != cudaSuccess) return e;
  if (M == 0) return cudaSuccess;
  return launch_norm<1>(x, nullptr, gamma, eps, M, K, nullptr, nullptr, absmax, nullptr, dev_err, s);
}

}  // namespace wql
