// norm.cu -- QRMSNorm fused with per-token dynamic int8 or fp8 quantisation, the same per-token
// quantisation of a row without the norm, and the calibration statistic used by weight smoothing ("LMDeploy W8A8 quantisation guide": QRMSNorm.forward,
// rms_norm_dynamic_quant, per_token_quant_int8 with scale = absmax / Q_MAX; int8 codes are rounded
// to integers (Q_MAX = 127), fp8 codes are the e4m3 cast (Q_MAX = 448); smoothing statistics are
// the per-channel absmax of the norm output).
//
// CTAs of 256 threads walk the token rows in groups of 64, 128 or 256 threads per row; each row is
// brought into shared memory by a bulk copy (several rows in flight per group) and held in
// registers while it is normalised.  The sum of squares uses a fixed order (chunk c of 8 elements
// belongs to lane c mod 256, which adds its elements in increasing k; the 256 lane sums are then
// folded pairwise (t, t+128), (t, t+64), ..., (t, t+1)), so int8 codes are reproducible bit for bit.
// Every float operation uses an explicitly rounded intrinsic; the one fused multiply-add (x * x + p)
// rounds exactly like the separate operations, since x * x is exact in fp32 for fp16 x.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace wql {
namespace {

constexpr int kNormThreads = 256;

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

// Rows in flight per row group (L groups per CTA, J chunks of 8 per lane): four for one group of
// up to 8192 elements, three otherwise.
__host__ __device__ constexpr int norm_slots(int l, int j, int mode) { return l == 1 && j <= 4 ? 4 : 3; }
__host__ __device__ constexpr int norm_rows_per_slot(int mode) { return mode_residual(mode) ? 2 : 1; }

// gamma in shared memory for many rows per CTA or long rows; CTAs per SM asked of the compiler
// (registers) -- both chosen by measurement (four CTAs of one 256-thread row per SM for rows up to
// 4096 elements, as many rows in flight as the residual mode's registers allow)
__host__ __device__ constexpr bool norm_gamma_in_smem(int l, int j, int mode) {
  return l > 1 || (j > 4 && !mode_residual(mode));
}
__host__ __device__ constexpr int norm_min_ctas(int l, int j, int mode) {
  return l == 1 ? (j <= 2 ? (mode_residual(mode) ? 3 : 4) : (j <= 4 || mode_residual(mode) ? 1 : 2))
                : (mode_residual(mode) ? 2 : 3);
}

// Low bytes of four ints, packed little-endian.
__device__ __forceinline__ uint32_t pack_s8x4(int c0, int c1, int c2, int c3) {
  const uint32_t lo = prmt((uint32_t)c0, (uint32_t)c1, 0x0040u), hi = prmt((uint32_t)c2, (uint32_t)c3, 0x0040u);
  return prmt(lo, hi, 0x5410u);
}

// A group of RT = 256 / L threads normalises one row; a CTA of 256 threads holds L groups, each with
// its own named barrier (ids 1..L; 0 is __syncthreads).  Fewer threads per row spread each row's
// fixed work -- two reductions, the divisions and the square root, which every warp evaluates --
// over more elements per thread (the kernel is bound by instruction issue).
template <int L>
struct RowGroup {
  static constexpr int kRT = kNormThreads / L;  // threads per row
  static constexpr int kW = kRT / 32;           // warps per row
};

// Named barrier of `count` threads that also returns whether any of them passed `pred` true.
__device__ __forceinline__ bool group_sync_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Sum of the 256 lane partials in the fixed order (t, t+128), (t, t+64), ..., (t, t+1).  Thread gt
// of the group holds lanes gt + RT i (i < L) and folds the levels with strides >= RT itself; every
// warp then evaluates the cross-warp levels (lane l from the partials l + 32 w, in exactly that
// order) and the five shuffle levels, so all threads get the same total as with one lane per
// thread.  The barrier also votes: it returns false in every thread of the group if `ok` is false in
// any of them.
template <int L>
__device__ __forceinline__ bool row_sum_vote(const float (&p)[L], bool ok, float* red, int gt, int bar, float& total) {
  constexpr int RT = RowGroup<L>::kRT, W = RowGroup<L>::kW;
  float v;
  if constexpr (L == 1) {
    v = p[0];
  } else if constexpr (L == 2) {
    v = __fadd_rn(p[0], p[1]);  // (gt, gt + 128)
  } else {
    static_assert(L == 4, "one, two or four lanes per thread");
    v = __fadd_rn(__fadd_rn(p[0], p[2]), __fadd_rn(p[1], p[3]));  // (gt, gt+128), (gt+64, gt+192); (gt, gt+64)
  }
  red[gt] = v;
  if (group_sync_or(bar, RT, !ok)) return false;
  const int lane = gt & 31;
  float x[W];
#pragma unroll
  for (int w = 0; w < W; ++w) x[w] = red[lane + 32 * w];
#pragma unroll
  for (int st = W / 2; st >= 1; st >>= 1)
#pragma unroll
    for (int w = 0; w < st; ++w) x[w] = __fadd_rn(x[w], x[w + st]);
  v = x[0];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
  total = __shfl_sync(0xffffffffu, v, 0);
  return true;
}

// Row maximum over the group: one more barrier, with a scratch area distinct from the sum's.
template <int L>
__device__ __forceinline__ float row_max(float v, float* redmax, int gt, int bar) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  if ((gt & 31) == 0) redmax[gt >> 5] = v;
  named_barrier_sync(bar, RowGroup<L>::kRT);
  float m = redmax[0];
#pragma unroll
  for (int w = 1; w < RowGroup<L>::kW; ++w) m = fmaxf(m, redmax[w]);
  return m;
}

// Quantising modes write (q, xs); MODE 1 writes the per-channel absmax of the norm output.  The
// residual modes add the residual first ("LMDeploy W8A8 quantisation guide", inference kernels: the
// residual fusion of rms_norm_dynamic_quant): h = fp16(fp32(x) + fp32(r)) is stored to h_out (the
// new residual; it may be the residual buffer itself) and normalised and quantised like x.
// Persistent CTAs of L row groups: group g of CTA b normalises rows G, G + S, ... with
// G = b L + g and S = gridDim.x L.  Its first thread keeps kNormSlots rows in flight with bulk
// copies into the group's shared-memory ring, so HBM reads continue through every row's
// reductions; a slot is refilled as soon as the group's threads have all read it (the first
// barrier of the row's sum).  Thread gt takes the 8-element chunks c = lane + 256 j of lanes
// lane = gt + RT i (i < L, j < J): chunk c belongs to lane c mod 256, as the fixed summation order
// requires.  gamma is kept as fp32, in registers when a thread has at most 32 elements of it and
// in shared memory otherwise (norm_gamma_in_smem).
template <int L, int J, int MODE>
__global__ void __launch_bounds__(kNormThreads, norm_min_ctas(L, J, MODE))
    qrmsnorm_kernel(const __half* __restrict__ x, const __half* residual, const __half* __restrict__ gamma, float eps,
                    int M, int K, uint8_t* __restrict__ q, float* __restrict__ xs, float* __restrict__ absmax,
                    __half* h_out, unsigned* err) {
  constexpr int RT = RowGroup<L>::kRT;
  constexpr int kNormSlots = norm_slots(L, J, MODE), kRowsPerSlot = norm_rows_per_slot(MODE);
  constexpr bool kResid = mode_residual(MODE);
  constexpr bool kNorm = !mode_no_norm(MODE);
  __shared__ float red[kNormThreads + 8 * L];  // [group][RT] lane partials, then [group][8] warp maxima
  __shared__ __align__(8) uint64_t full[L][kNormSlots];
  extern __shared__ __align__(16) uint8_t dsm[];  // [L][kNormSlots][kRowsPerSlot x 2K] rows, then gamma (fp32)
  const int g = threadIdx.x / RT, gt = threadIdx.x % RT, bar = 1 + g;
  const int nchunks = K >> 3;
  const uint32_t row_bytes = 2u * (uint32_t)K;
  const uint32_t slot_bytes = kRowsPerSlot * row_bytes;
  uint8_t* rows = dsm + (size_t)g * kNormSlots * slot_bytes;
  const float* gsm = reinterpret_cast<const float*>(dsm + (size_t)L * kNormSlots * slot_bytes);
  float* gred = red + g * RT;
  float* gmax = red + kNormThreads + 8 * g;
  const int first = (int)blockIdx.x * L + g, stride = (int)gridDim.x * L;
  const int nrows = M > first ? (M - 1 - first) / stride + 1 : 0;
  auto issue = [&](int j) {  // row j of this group (and its residual row) into slot j % kNormSlots
    const int s = j % kNormSlots;
    const size_t off = (size_t)(first + (size_t)j * stride) * K;
    mbar_arrive_expect_tx(&full[g][s], slot_bytes);
    bulk_load(rows + (size_t)s * slot_bytes, x + off, row_bytes, &full[g][s]);
    if constexpr (kResid) bulk_load(rows + (size_t)s * slot_bytes + row_bytes, residual + off, row_bytes, &full[g][s]);
  };
  if (gt == 0) {
    for (int s = 0; s < kNormSlots; ++s) mbar_init(&full[g][s], 1);
    fence_mbarrier_init();
  }
  // gamma, read once per CTA as fp32: into shared memory, or into this thread's registers
  constexpr bool kGammaSmem = norm_gamma_in_smem(L, J, MODE);
  float gfr[kGammaSmem ? 1 : L][kGammaSmem ? 1 : J][8];
  if constexpr (kNorm && !kGammaSmem) {
    const uint4* gr = reinterpret_cast<const uint4*>(gamma);
#pragma unroll
    for (int i = 0; i < L; ++i)
#pragma unroll
      for (int jj = 0; jj < J; ++jj) {
        const int c = gt + RT * i + kNormThreads * jj;
        if (c < nchunks) {
          const uint4 gv = __ldg(gr + c);
          const __half* gh = reinterpret_cast<const __half*>(&gv);
#pragma unroll
          for (int e = 0; e < 8; ++e) gfr[i][jj][e] = __half2float(gh[e]);
        }
      }
  }
  if constexpr (kNorm && kGammaSmem) {
    float* gw = const_cast<float*>(gsm);
    const uint4* gr = reinterpret_cast<const uint4*>(gamma);
    for (int c = threadIdx.x; c < nchunks; c += kNormThreads) {
      const uint4 gv = __ldg(gr + c);
      const __half* gh = reinterpret_cast<const __half*>(&gv);
      float4 a, b;
      a.x = __half2float(gh[0]), a.y = __half2float(gh[1]), a.z = __half2float(gh[2]), a.w = __half2float(gh[3]);
      b.x = __half2float(gh[4]), b.y = __half2float(gh[5]), b.z = __half2float(gh[6]), b.w = __half2float(gh[7]);
      reinterpret_cast<float4*>(gw)[2 * c] = a;
      reinterpret_cast<float4*>(gw)[2 * c + 1] = b;
    }
  }
  __syncthreads();
  // x comes from the preceding kernel, which may also still read q and xs
  grid_dependency_wait();
  if (gt == 0) {
    for (int j = 0; j < nrows && j < kNormSlots; ++j) issue(j);
    if (g == 0) grid_dependents_launch();  // the next kernel's copies now queue behind these
  }

  int j = 0;
  for (; j < nrows; ++j) {
    const int m = first + j * stride;
    const int s = j % kNormSlots;
    // Every thread waits; the row sum's barrier votes, so that all threads leave together if a wait
    // ever expires (the values read from an unfinished slot are then discarded).
    const bool ok = mbar_wait_bounded(&full[g][s], (j / kNormSlots) & 1);
    const uint4* xr = reinterpret_cast<const uint4*>(rows + (size_t)s * slot_bytes);
    float yv[L][J][8];  // x (or x + r as fp16), then the normalised row
    uint4 hv[kResid ? L : 1][kResid ? J : 1];  // the new residual, stored once the row's wait is confirmed
    float p[L];
#pragma unroll
    for (int i = 0; i < L; ++i) {
      p[i] = 0.f;
#pragma unroll
      for (int jj = 0; jj < J; ++jj) {
        const int c = gt + RT * i + kNormThreads * jj;
        if (c < nchunks) {
          uint4 xv = xr[c];
          if constexpr (kResid) {
            const uint4 rv = reinterpret_cast<const uint4*>(rows + (size_t)s * slot_bytes + row_bytes)[c];
            const __half* xh = reinterpret_cast<const __half*>(&xv);
            const __half* rh = reinterpret_cast<const __half*>(&rv);
            __align__(16) __half hh[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) hh[e] = __float2half_rn(__fadd_rn(__half2float(xh[e]), __half2float(rh[e])));
            hv[i][jj] = *reinterpret_cast<const uint4*>(hh);
            xv = hv[i][jj];
          }
          const __half* h = reinterpret_cast<const __half*>(&xv);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float v = __half2float(h[e]);
            yv[i][jj][e] = v;
            // v * v is exact in fp32 (fp16 has an 11-bit significand), so the fused multiply-add
            // rounds exactly as the separate product and sum do
            if constexpr (kNorm) p[i] = __fmaf_rn(v, v, p[i]);
          }
        }
      }
    }
    // the slot was read through the generic proxy and the group's first thread refills it with a
    // bulk copy (async proxy) after the next barrier: a proxy fence orders the reads before that write
    fence_proxy_async_smem();
    float ss;
    if (!row_sum_vote<L>(p, ok, gred, gt, bar, ss)) {
      if (gt == 0) report_error(err, kErrTimeoutFull);
      break;
    }
    // every thread of the group has read slot s (it passed the sum's barrier): refill it
    if (gt == 0 && j + kNormSlots < nrows) issue(j + kNormSlots);
    if constexpr (kResid) {
#pragma unroll
      for (int i = 0; i < L; ++i)
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
          const int c = gt + RT * i + kNormThreads * jj;
          if (c < nchunks) *reinterpret_cast<uint4*>(h_out + (size_t)m * K + 8 * c) = hv[i][jj];
        }
    }
    float amax = 0.f;
    if constexpr (kNorm) {
      const float mean = __fdiv_rn(ss, (float)K);
      const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
#pragma unroll
      for (int i = 0; i < L; ++i)
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
          const int c = gt + RT * i + kNormThreads * jj;
          if (c < nchunks) {
            float gf[8];
            if constexpr (kGammaSmem) {
              const float4 g0 = reinterpret_cast<const float4*>(gsm)[2 * c];
              const float4 g1 = reinterpret_cast<const float4*>(gsm)[2 * c + 1];
              gf[0] = g0.x, gf[1] = g0.y, gf[2] = g0.z, gf[3] = g0.w, gf[4] = g1.x, gf[5] = g1.y, gf[6] = g1.z,
              gf[7] = g1.w;
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) gf[e] = gfr[i][jj][e];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float yy = __fmul_rn(__fmul_rn(yv[i][jj][e], r), gf[e]);
              yv[i][jj][e] = yy;
              amax = fmaxf(amax, fabsf(yy));
            }
          }
        }
    } else {  // per-token quantisation of the row itself
#pragma unroll
      for (int i = 0; i < L; ++i)
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
          const int c = gt + RT * i + kNormThreads * jj;
          if (c < nchunks) {
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(yv[i][jj][e]));
          }
        }
    }

    if (MODE == 1) {
#pragma unroll
      for (int i = 0; i < L; ++i)
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
          const int c = gt + RT * i + kNormThreads * jj;
          if (c < nchunks) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              atomicMax(reinterpret_cast<int*>(absmax) + 8 * c + e, __float_as_int(fabsf(yv[i][jj][e])));
          }
        }
      named_barrier_sync(bar, RT);  // the lane partials are read by every warp before the next row writes them
      continue;
    }

    const float rowmax = row_max<L>(amax, gmax, gt, bar);
    const float scale = rowmax == 0.f ? 1.0f : __fdiv_rn(rowmax, mode_fp8(MODE) ? 448.0f : 127.0f);
    const float inv = __fdiv_rn(1.0f, scale);
    if (gt == 0) xs[m] = scale;
    uint8_t* qr = q + (size_t)m * K;
#pragma unroll
    for (int i = 0; i < L; ++i)
#pragma unroll
      for (int jj = 0; jj < J; ++jj) {
        const int c = gt + RT * i + kNormThreads * jj;
        const float* yy = yv[i][jj];
        if (mode_fp8(MODE) && c < nchunks) {
          const float y0[4] = {yy[0], yy[1], yy[2], yy[3]};
          const float y1[4] = {yy[4], yy[5], yy[6], yy[7]};
          *reinterpret_cast<uint2*>(qr + 8 * c) = make_uint2(e4m3x4_div(y0, scale, inv), e4m3x4_div(y1, scale, inv));
        } else if (c < nchunks) {
          int k8[8];
          bool exact = false;
#pragma unroll
          for (int e = 0; e < 8; ++e) k8[e] = quant_fast(yy[e], inv, exact);
          if (exact) {  // rare: some element lies within 5e-5 of a rounding tie
#pragma unroll
            for (int e = 0; e < 8; ++e) k8[e] = quant_exact(yy[e], scale, inv);
          }
          *reinterpret_cast<uint2*>(qr + 8 * c) =
              make_uint2(pack_s8x4(k8[0], k8[1], k8[2], k8[3]), pack_s8x4(k8[4], k8[5], k8[6], k8[7]));
        }
      }
  }
  // Leave no copy in flight: after an expired wait, wait (bounded) for the rows still issued.
  if (j < nrows && gt == 0) {
    const int issued = nrows < j + kNormSlots ? nrows : j + kNormSlots;
    for (int i = j; i < issued; ++i)
      if (!mbar_wait_bounded(&full[g][i % kNormSlots], (i / kNormSlots) & 1)) {
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

template <int L, int J, int MODE>
cudaError_t launch_rows(const __half* x, const __half* residual, const __half* gamma, float eps, int M, int K,
                        uint8_t* q, float* xs, float* absmax, __half* h_out, unsigned* err, cudaStream_t s) {
  auto kern = qrmsnorm_kernel<L, J, MODE>;
  // the row groups' rings, then gamma as fp32 if it lives in shared memory
  const size_t smem = (size_t)L * norm_slots(L, J, MODE) * norm_rows_per_slot(MODE) * 2 * K +
                      (mode_no_norm(MODE) || !norm_gamma_in_smem(L, J, MODE) ? 0 : (size_t)4 * K);
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
  const long long need = ((long long)M + L - 1) / L;  // L rows per CTA at a time
  const dim3 grid((unsigned)(need < cap ? need : cap)), block(kNormThreads);
  return launch_pdl(kern, grid, block, smem, s, x, residual, gamma, eps, M, K, q, xs, absmax, h_out, err);
}

template <int MODE>
cudaError_t launch_norm(const uint16_t* x, const uint16_t* residual, const uint16_t* gamma, float eps, int M, int K,
                        uint8_t* q, float* xs, float* absmax, uint16_t* h_out, unsigned* err, cudaStream_t s) {
  const __half* xh = reinterpret_cast<const __half*>(x);
  const __half* rh = reinterpret_cast<const __half*>(residual);
  const __half* gh = reinterpret_cast<const __half*>(gamma);
  __half* hh = reinterpret_cast<__half*>(h_out);
  // J chunks of 8 elements per lane.  Many rows: rows of up to 2048 / 4096 elements take 64 / 128
  // threads, which spreads each row's fixed work over more elements (M = 4096: K = 4096 18.1 ->
  // 16.2 us, K = 2048 13.0 -> 9.4 us).  Few rows, or the residual modes (which hold twice the data
  // per element), keep 256 threads per row: shorter rows in flight (M = 512, K = 4096: 4.1 us with
  // 256 threads, 5.0 with 128; add + norm at M = 4096: 22.5 against 29.0).
  const int cpl = (K + 2047) / 2048;
  const bool grouped = M >= 2048 && !mode_residual(MODE);
  if (cpl <= 1) {
    if (grouped) return launch_rows<4, 1, MODE>(xh, rh, gh, eps, M, K, q, xs, absmax, hh, err, s);
    return launch_rows<1, 1, MODE>(xh, rh, gh, eps, M, K, q, xs, absmax, hh, err, s);
  }
  if (cpl <= 2) {
    if (grouped) return launch_rows<2, 2, MODE>(xh, rh, gh, eps, M, K, q, xs, absmax, hh, err, s);
    return launch_rows<1, 2, MODE>(xh, rh, gh, eps, M, K, q, xs, absmax, hh, err, s);
  }
  if (cpl <= 4) return launch_rows<1, 4, MODE>(xh, rh, gh, eps, M, K, q, xs, absmax, hh, err, s);
  return launch_rows<1, 8, MODE>(xh, rh, gh, eps, M, K, q, xs, absmax, hh, err, s);
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
