// fp8_prefill.cu -- the fp8 (e4m3) variant of the SmoothQuant W8A8 GEMM for prefill-shaped calls,
// on the tcgen05 tensor cores ("LMDeploy W8A8 quantisation guide": quant_dtype fp8 is
// float8_e4m3fn; matmul_kernel_dynamic_quant takes an fp32 accumulator for floating-point inputs,
// then c = c * rms_scale * linear_scale, rounded to fp16; its _linear_add variant adds a bias and a
// residual).
//
// Both operands are e4m3 codes, which kind::f8f6f4 reads straight from shared memory, so nothing is
// converted: TMA brings 128-byte-swizzled tiles of the weights qw [N, K] (128 output channels, the
// MMA's M: "swap AB") and of the activation codes q [M, K] (BN tokens, the MMA's N), 128 k per stage,
// and one thread issues four K = 32 MMAs per stage.  Warp roles: warp 0 the TMA producer, warp 1 the
// MMA issuer (and TMEM owner), warps 2-5 the epilogue.  Two TMEM accumulators of BN columns alternate
// between tiles, so a tile's epilogue overlaps the next tile's MMAs.  Persistent CTAs walk the tiles,
// channel tiles fastest (CTAs running at the same time share the token tile).
//
// The epilogue stages its output through shared memory: each epilogue warp owns 32 channels and
// works on 32 tokens at a time, in a 32 x 32 fp16 box.  When a residual is fused, TMA loads the
// tile's residual boxes ahead (all four with one CTA per SM, two with two) while the tile's MMAs
// run, and the outputs replace them in place; a TMA store writes each finished box to y.  So the
// epilogue issues no scalar global loads or stores on its critical path (the residual read through
// scalar loads doubled the kernel's time: ncu, M = N = K = 4096, 82.5 -> 161 us).
//
// One CTA's MMA thread keeps the tensor pipe busy only about 40 % of the time (ncu, M = N = K = 4096:
// its barrier round trips and commits leave gaps that deeper stages or 256-k stages do not close).
// When there are more tiles than SMs, two CTAs of three stages share each SM and fill each other's
// gaps: M = 8192, N = 4096: 143 -> 107 us; M = 4096, N = 11008: 184 -> 144 us.
#include <atomic>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace wql {
namespace {

constexpr int kBK = 128;  // k per stage (bytes of an e4m3 row): four K = 32 MMAs
constexpr int kBM = 128;  // output channels per tile (MMA M)
constexpr int kProducerWarp = 0, kMmaWarp = 1, kEpiWarp0 = 2, kEpiWarps = 4;
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;

template <int BN, int CTAS>
struct FLayout {
  static constexpr int kWBytes = kBM * kBK;  // 128 channel rows x 128 B, 128-byte swizzle
  static constexpr int kXBytes = BN * kBK;   // BN token rows x 128 B
  static constexpr int kStage = kWBytes + kXBytes;
  static_assert(BN == 64 || BN == 128, "token tiles of 64 or 128");
  static constexpr int kStages = CTAS == 2 ? 3 : (BN == 128 ? 6 : 8);  // 192 KB of stages with one CTA
  static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators of BN fp32 columns
  static constexpr int kBox = 32 * 32 * 2;                     // one 32 tokens x 32 channels fp16 box
  static constexpr int kBufs = CTAS == 2 ? 2 : 4;              // output boxes per epilogue warp
  static constexpr int kOffOut = kStages * kStage;             // [epilogue warp][kBufs] boxes
  static constexpr int kOffBar = kOffOut + kEpiWarps * kBufs * kBox;
  static constexpr int kBarBytes = (2 * kStages + 5 + kBufs * kEpiWarps) * 8 + 16;
  // Two CTAs per SM leave no room for aligning the dynamic shared memory by hand: the kernel then
  // relies on its base being 1024-byte aligned (it is placed right after the reserved 1 KB), checks
  // it, and reports kErrSmemAlign instead of running if it is not.
  static constexpr int kSlack = CTAS == 2 ? 0 : 1024;
  static constexpr int kBytes = kOffBar + kBarBytes + kSlack;
  static_assert(kStage % 1024 == 0, "stages keep the 1024-byte alignment of the swizzle atoms");
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation");
  static_assert(kBytes <= (CTAS == 2 ? 113 : 227) * 1024, "shared memory budget");
  static_assert(CTAS == 1 || 2 * kTmemCols <= 512, "TMEM budget of two CTAs per SM");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int BN, int CTAS>
__global__ void __launch_bounds__(kThreads, CTAS)
    fp8_prefill_kernel(const __grid_constant__ CUtensorMap tm_x,  // q e4m3 [M][K], box {128, BN}, SW128
                       const __grid_constant__ CUtensorMap tm_w,  // qw e4m3 [N][K], box {128, 128}, SW128
                       const __grid_constant__ CUtensorMap tm_y,  // y fp16 [M][N], box {32, 32}
                       const __grid_constant__ CUtensorMap tm_r,  // residual fp16 [M][N], box {32, 32}
                       const float* __restrict__ xs, const float* __restrict__ ws, int M, int N, int K,
                       float* __restrict__ acc_out, EpilogueAdd ea, unsigned* err) {
  using L = FLayout<BN, CTAS>;
  constexpr int kStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  if (smem - smem_raw > L::kSlack) {  // uniform over the CTA: before any barrier or TMEM use
    if (threadIdx.x == 0) report_error(err, kErrSmemAlign);
    return;
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* empty = full + kStages;     // the stage's MMAs have completed
  uint64_t* accfull = empty + kStages;  // [2] accumulator holds a finished tile
  uint64_t* accempty = accfull + 2;     // [2] epilogue has read the accumulator
  uint64_t* finalbar = accempty + 2;
  uint64_t* rfull = finalbar + 1;       // [epilogue warp][kBufs] residual box landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rfull + L::kBufs * kEpiWarps);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntn = (N + kBM - 1) / kBM;
  const int ntiles = ntn * ((M + BN - 1) / BN);
  const int nkb = (K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], kEpiWarps);
    }
    mbar_init(finalbar, 1);
    for (int i = 0; i < L::kBufs * kEpiWarps; ++i) mbar_init(&rfull[i], 1);
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_w);
      grid_dependency_wait();
      int stage = 0, phase = 0, issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const int nt = tile % ntn, mt = tile / ntn;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1)) {
            report_error(err, kErrTimeoutEmpty);
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * L::kStage;
          mbar_arrive_expect_tx(&full[stage], L::kStage);
          tma_load_2d(st, &tm_w, &full[stage], kb * kBK, nt * kBM);
          tma_load_2d(st + L::kWBytes, &tm_x, &full[stage], kb * kBK, mt * BN);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // leave no copy in flight: wait (bounded) for the last stages issued
      for (int i = 0; i < kStages && i < issued; ++i) {
        stage = stage == 0 ? kStages - 1 : stage - 1;
        if (stage == kStages - 1) phase ^= 1;
        if (!mbar_wait_bounded(&full[stage], phase)) {
          report_error(err, kErrTimeoutDrain);
          break;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_e4m3(kBM, BN);
      int stage = 0, phase = 0, tcount = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++tcount) {
        const int b = tcount & 1;
        if (!mbar_wait_bounded(&accempty[b], ((tcount >> 1) & 1) ^ 1)) {
          report_error(err, kErrTimeoutMma);
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + b * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase)) {
            report_error(err, kErrTimeoutMma);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // the stage's descriptors differ only in the start address field (bits 0-13, addr >> 4;
          // shared-memory addresses stay below 2^18, so adding to it never carries): 32 bytes per
          // K = 32 step along the 128-byte rows
          const uint32_t st = smem_u32(smem + stage * L::kStage);
          const uint64_t adesc0 = umma_sdesc_sw128(st, 16, 1024);
          const uint64_t bdesc0 = umma_sdesc_sw128(st + L::kWBytes, 16, 1024);
#pragma unroll
          for (int s = 0; s < kBK / 32; ++s)
            umma_f8f6f4(d_tmem, adesc0 + 2 * s, bdesc0 + 2 * s, idesc, (kb > 0 || s > 0) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&accfull[b]);
      }
      umma_commit(finalbar);
      if (!mbar_wait_bounded(finalbar, 0)) report_error(err, kErrTimeoutDrain);
    }
  } else {
    // ---------------- epilogue: TMEM lane = output channel, column = token ----------------
    const int ew = warp - kEpiWarp0;
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    BoxStage<L::kBufs> out;
    out.init(reinterpret_cast<__half*>(smem + L::kOffOut + ew * L::kBufs * L::kBox), rfull + ew * L::kBufs, &tm_y,
             &tm_r, ea.residual != nullptr);
    int tcount = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++tcount) {
      const int nt = tile % ntn, mt = tile / ntn;
      const int b = tcount & 1;
      const int n0 = nt * kBM + quad * 32, n = n0 + lane;
      const float wn = n < N ? ws[n] : 0.f;
      const float bn = (ea.bias && n < N) ? __half2float(ea.bias[n]) : 0.f;
      out.begin(n0, mt * BN, BN / 32, lane);  // residual boxes land while the tile's MMAs run
      if (!mbar_wait_warp(&accfull[b], (tcount >> 1) & 1)) {
        report_error(err, kErrTimeoutMma);
        break;
      }
      tc_fence_after_sync();
#pragma unroll 1
      for (int j = 0; j < BN / 32; ++j) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(lane_base + b * BN + 32 * j, r);
        const int mbase = mt * BN + 32 * j;
        const float xl = mbase + lane < M ? xs[mbase + lane] : 0.f;
        tmem_ld_wait();
        __half* bx = out.acquire(j, lane);
        if (!bx) {
          report_error(err, kErrTimeoutFull);
          ok = false;
          break;
        }
        // row k of the box = token mbase + k; lane = channel: 32 lanes touch 64 contiguous bytes
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float xm = __shfl_sync(0xffffffffu, xl, k);
          const float c = __uint_as_float(r[k]);
          const float rr = out.has_res ? __half2float(bx[k * 32 + lane]) : 0.f;
          bx[k * 32 + lane] = __float2half_rn(add_terms(__fmul_rn(__fmul_rn(c, xm), wn), ea, bn, rr));
          if (acc_out && n < N && mbase + k < M) acc_out[(size_t)(mbase + k) * N + n] = c;
        }
        out.store(j, bx, lane);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[b]);
    }
    if (!out.finish(lane)) report_error(err, kErrTimeoutDrain);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, L::kTmemCols);
}

template <int BN, int CTAS>
cudaError_t launch_f(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, const CUtensorMap& tr,
                     const float* xs, const float* ws, int M, int N, int K, float* acc_out, EpilogueAdd ea,
                     unsigned* dev_err, cudaStream_t stream) {
  using L = FLayout<BN, CTAS>;
  auto kern = fp8_prefill_kernel<BN, CTAS>;
  static std::atomic<bool> attr_set[64];  // per device; racing first calls set the same attribute
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const int ntiles = ((N + kBM - 1) / kBM) * ((M + BN - 1) / BN);
  const int grid = ntiles < CTAS * num_sms() ? ntiles : CTAS * num_sms();
  kern<<<grid, kThreads, L::kBytes, stream>>>(tx, tw, ty, tr, xs, ws, M, N, K, acc_out, ea, dev_err);
  return cudaGetLastError();
}

template <int BN>
cudaError_t launch_bn(const void* q, const void* qw, const float* xs, const float* ws, int M, int N, int K, __half* y,
                      float* acc_out, EpilogueAdd ea, unsigned* dev_err, cudaStream_t stream, std::string* err) {
  CUtensorMap tx, tw, ty, tr;
  if (!make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q, K, M, (uint64_t)K, kBK, BN, CU_TENSOR_MAP_SWIZZLE_128B,
                    err) ||
      !make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qw, K, N, (uint64_t)K, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B,
                    err) ||
      !make_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, y, N, M, (uint64_t)N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE,
                    err) ||
      (ea.residual && !make_tmap_2d(&tr, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ea.residual, N, M, (uint64_t)N * 2, 32, 32,
                                    CU_TENSOR_MAP_SWIZZLE_NONE, err))) {
    return cudaErrorInvalidValue;
  }
  if (!ea.residual) tr = ty;  // not read
  // two CTAs per SM only when every SM gets at least one tile: with fewer tiles than SMs the block
  // scheduler may pair CTAs on some SMs while others stay idle (M = 512, N = 4096: 19.6 -> 20.5 us)
  const long long ntiles = (long long)((N + kBM - 1) / kBM) * ((M + BN - 1) / BN);
  if (ntiles > num_sms()) return launch_f<BN, 2>(tx, tw, ty, tr, xs, ws, M, N, K, acc_out, ea, dev_err, stream);
  return launch_f<BN, 1>(tx, tw, ty, tr, xs, ws, M, N, K, acc_out, ea, dev_err, stream);
}

}  // namespace

// Token tile for an fp8 GEMM of M tokens: 64 up to 64 tokens, else 128.  A 256-token tile (fewer,
// longer tiles, four stages) measured slower at every shape tried on GB300 (K = 4096, N = 4096 and
// 11008, M = 128 .. 8192: e.g. M = 4096, N = 11008: 198 vs 182 us; M = 512, N = 4096: 28.4 vs 19.8 us).
// When 128-token tiles would leave SMs idle but 64-token tiles outnumber the SMs, the smaller tiles
// run two CTAs per SM instead.
int fp8_prefill_tile_n(int M, int N) {
  if (M <= 64) return 64;
  const long long ntn = (N + kBM - 1) / kBM, sms = num_sms();
  if (ntn * ((M + 127) / 128) <= sms && ntn * ((M + 63) / 64) > sms) return 64;
  return 128;
}

cudaError_t launch_fp8_prefill(const uint8_t* q, const float* xs, const uint8_t* qw, const float* ws, int M, int K,
                               int N, uint16_t* y, float* acc_out, const uint16_t* bias, const uint16_t* residual,
                               unsigned* dev_err, cudaStream_t stream, std::string* err) {
  const EpilogueAdd ea{reinterpret_cast<const __half*>(bias), reinterpret_cast<const __half*>(residual)};
  __half* yh = reinterpret_cast<__half*>(y);
  if (fp8_prefill_tile_n(M, N) == 64) return launch_bn<64>(q, qw, xs, ws, M, N, K, yh, acc_out, ea, dev_err, stream, err);
  return launch_bn<128>(q, qw, xs, ws, M, N, K, yh, acc_out, ea, dev_err, stream, err);
}

}  // namespace wql
