// w8a8_prefill.cu -- SmoothQuant W8A8 GEMM for prefill-shaped calls on the tcgen05 tensor cores
// ("LMDeploy W8A8 quantisation guide", QLinear.forward / matmul_kernel_dynamic_quant: int8 x int8
// products summed in int32, then c = c * rms_scale * linear_scale in fp32, rounded to fp16).
//
// GB300's tcgen05 has no int8 kind, and int8 values are exact in fp16, so both operands run on
// kind::f16 as exact fp16 integers:
//   * a pre-pass converts the activation codes q [M, K] to fp16 in the caller's workspace (TMA then
//     reads them like any fp16 operand);
//   * warps 2-9 convert each 128 x 64 int8 weight tile to fp16 and write it straight into tensor
//     memory, which the MMA reads as its A operand (weights are the 128-row operand: "swap AB").
//     A thread owns one output channel, i.e. one TMEM lane, and half of the tile's 64 k: the int8
//     weight rows are K-contiguous, so its 64 codes are four 16-byte shared-memory loads (the tile
//     arrives with a 128-byte swizzle, which spreads a warp's rows over all banks).  Keeping the
//     fp16 operand out of shared memory removes two thirds of the shared-memory traffic per stage;
//   * exactness: |product| <= 128 * 128 = 2^14 (both codes may be -128), so any partial sum of row
//     m is an integer of magnitude <= 128 * sum_k |q[m, k]|.  When that bound stays within 2^24 for
//     every row (the conversion pre-pass records the largest row L1 norm of each of its blocks;
//     typical per-token codes at K = 4096 stay near 2^16), one fp32 accumulator takes the whole of
//     K exactly, and the TMEM
//     the chunk scheme needs holds more A slots instead (4 against 2 at 128 tokens).  Otherwise each
//     accumulator covers at most 1024 k, which bounds every partial sum by 2^24: the MMA thread
//     alternates two TMEM chunk accumulators, and the epilogue warps turn each finished chunk into
//     int32 and add it to an int32 running sum kept in TMEM, so the MMAs never wait for them.
//     Either way the tile yields the exact acc (written to acc_out if requested) and
//     y = fp16((float(acc) * xs[m]) * ws[n]);
//   * each epilogue warp owns 32 channels and writes y in 32-token boxes staged through shared memory
//     and stored by TMA; a fused residual arrives the same way: TMA loads all of the tile's residual
//     boxes while its last chunk's MMAs run (scalar residual loads on the epilogue's path made the
//     M = 4096, N = 11008 block 1.9x slower).
#include <atomic>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace wql {
namespace {

constexpr int kBK = 128;        // k per stage (bytes of a weight row): 8 MMAs per barrier round trip
constexpr int kBM = 128;        // output channels per tile (MMA M)
constexpr int kChunkKB = 8;     // stages per exact chunk: 8 x 128 = 1024 k
constexpr int kOneChunkL1 = (1 << 24) / 128;  // largest row L1 norm for which one chunk is exact
constexpr int kPrepassMaxBlocks = 4096;        // the pre-pass writes one row-norm maximum per block
constexpr int kProducerWarp = 0, kMmaWarp = 1, kCvWarp0 = 2, kCvWarps = 8, kEpiWarp0 = 10, kEpiWarps = 4;
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;

template <int BN>
struct QLayout {
  static constexpr int kXBox = BN * 128;         // BN token rows x 64 k fp16 (from the workspace)
  static constexpr int kXBytes = 2 * kXBox;      // two 64-k boxes per stage
  static constexpr int kWBytes = kBM * kBK;      // 128 rows x 128 int8, 128-byte swizzle
  static constexpr int kOffW = kXBytes;
  static constexpr int kStage = (kOffW + kWBytes + 1023) / 1024 * 1024;
  static constexpr int kStages = BN >= 128 ? 4 : 6;
  static constexpr uint32_t kTx = kXBytes + kWBytes;
  // TMEM columns: [0, BN) and [BN, 2 BN) chunk accumulators, [2 BN, 3 BN) int32 running sum, then
  // the fp16 A operand: kASlots slots of 64 columns (128 k) each
  static constexpr uint32_t kTmemCols = 512;
  // chunked mode: [2 BN, 3 BN) int32 running sum, then kChunkSlots A slots; one-chunk mode:
  // kOneSlots A slots from 2 BN
  static constexpr uint32_t kSumCol = 2 * BN;
  static constexpr int kChunkSlots = BN >= 128 ? 2 : 4;
  static constexpr int kOneSlots = (kTmemCols - 2 * BN) / 64;
  static constexpr int kASlots = kOneSlots;  // the larger ring (barrier count)
  static_assert(3 * BN + 64 * kChunkSlots <= kTmemCols && 2 * BN + 64 * kOneSlots <= kTmemCols, "TMEM budget");
  static constexpr int kBox = 32 * 32 * 2;  // one 32 tokens x 32 channels fp16 output box
  static constexpr int kBufs = 4;           // output boxes per epilogue warp: a whole tile's
  static constexpr int kOffOut = kStages * kStage;  // [epilogue warp][kBufs] boxes
  static constexpr int kOffBar = kOffOut + kEpiWarps * kBufs * kBox;
  static constexpr int kBarBytes = (2 * kStages + kASlots + 6 + kBufs * kEpiWarps) * 8 + 16;
  static constexpr int kBytes = kOffBar + kBarBytes + 1024;
  // a converter waits for the stage release of block i - kASlots before reusing its A slot: that
  // barrier is then never a phase ahead
  static_assert(kStages >= kASlots, "ring depths");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// int8 codes [M][K] -> exact fp16 [M][K], and per block the largest row L1 norm sum_k |q| among its
// rows (which decides whether one fp32 accumulator takes the whole of K exactly).  One warp per row,
// 16 codes per lane and step; K a multiple of 16 and both pointers 16-byte aligned.
__global__ void __launch_bounds__(256) i8_to_f16_rows_kernel(const int8_t* __restrict__ q, __half* __restrict__ out,
                                                             int* __restrict__ blockmax, int M, int K) {
  __shared__ int wmax[8];
  const int lane = threadIdx.x & 31;
  const int k16 = K / 16;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  unsigned rmax = 0;
  for (long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < M; row += nwarps) {
    const uint4* src = reinterpret_cast<const uint4*>(q + row * K);
    uint4* dst = reinterpret_cast<uint4*>(out + row * K);
    unsigned l1 = 0;
#pragma unroll 4
    for (int i = lane; i < k16; i += 32) {  // unrolled: several 16-byte loads in flight per lane
      const uint4 v = __ldg(src + i);
      uint4 a, b;
      i8x4_to_f16x2x2(v.x, a.x, a.y);
      i8x4_to_f16x2x2(v.y, a.z, a.w);
      i8x4_to_f16x2x2(v.z, b.x, b.y);
      i8x4_to_f16x2x2(v.w, b.z, b.w);
      dst[2 * i] = a;
      dst[2 * i + 1] = b;
      // per-byte |q| (0x80, i.e. -128, reads as the unsigned byte 128), summed by byte
      l1 += __vsadu4(__vabs4(v.x), 0u) + __vsadu4(__vabs4(v.y), 0u) + __vsadu4(__vabs4(v.z), 0u) +
            __vsadu4(__vabs4(v.w), 0u);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    rmax = l1 > rmax ? l1 : rmax;
  }
  if (lane == 0) wmax[threadIdx.x >> 5] = (int)rmax;
  __syncthreads();
  if (threadIdx.x == 0) {
    int b = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) b = wmax[w] > b ? wmax[w] : b;
    blockmax[blockIdx.x] = b;
  }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    w8a8_prefill_kernel(const __grid_constant__ CUtensorMap tm_x,  // fp16 codes [M][K], box {64, BN}, SW128
                        const __grid_constant__ CUtensorMap tm_w,  // qw int8 [N][K], box {64, 128}
                        const float* __restrict__ xs, const float* __restrict__ ws, int M, int N, int K,
                        const __grid_constant__ CUtensorMap tm_y,  // y fp16 [M][N], box {32, 32}
                        const __grid_constant__ CUtensorMap tm_r,  // residual fp16 [M][N], box {32, 32}
                        int32_t* __restrict__ acc_out, EpilogueAdd ea,
                        const int* __restrict__ blockmax,  // [nbm] largest row L1 norms of q (pre-pass)
                        int nbm, unsigned* err) {
  using L = QLayout<BN>;
  constexpr int kStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* empty = full + kStages;     // MMAs done with the stage (and with the blocks before it)
  uint64_t* afull = empty + kStages;    // [kASlots] A slot written to TMEM
  uint64_t* accfull = afull + L::kASlots;  // [2] chunk accumulators
  uint64_t* accempty = accfull + 2;     // [2]
  uint64_t* finalbar = accempty + 2;
  uint64_t* modebar = finalbar + 1;     // the accumulation mode is known
  uint64_t* rfull = modebar + 1;        // [epilogue warp][kBufs] residual box landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rfull + L::kBufs * kEpiWarps);
  int* mode_smem = reinterpret_cast<int*>(tmem_slot + 1);  // [0] max row L1 norm, [1] one-chunk mode

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntn = (N + kBM - 1) / kBM;
  const int ntm = (M + BN - 1) / BN;
  const int ntiles = ntn * ntm;
  const int nkb = (K + kBK - 1) / kBK;
  const int nchunks = (nkb + kChunkKB - 1) / kChunkKB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < L::kASlots; ++a) mbar_init(&afull[a], kCvWarps);  // one arrival per converter warp
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], kEpiWarps);
    }
    mbar_init(finalbar, 1);
    mbar_init(modebar, 1);
    mode_smem[0] = 0;
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
          mbar_arrive_expect_tx(&full[stage], L::kTx);
          tma_load_2d(st, &tm_x, &full[stage], kb * kBK, mt * BN);
          tma_load_2d(st + L::kXBox, &tm_x, &full[stage], kb * kBK + 64, mt * BN);
          tma_load_2d(st + L::kOffW, &tm_w, &full[stage], kb * kBK, nt * kBM);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
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
      constexpr uint32_t idesc = umma_idesc_f16(kBM, BN, /*A K-major*/ 0, /*B K-major*/ 0);
      int stage = 0, phase = 0, aslot = 0, aph = 0, cseq = 0;  // cseq counts chunks over all tiles
      bool ok = mbar_wait_bounded(modebar, 0);
      if (!ok) report_error(err, kErrTimeoutMma);
      const bool one = ok && mode_smem[1] != 0;
      const int chunk_kb = one ? nkb : kChunkKB, nch = one ? 1 : nchunks;
      const int nslots = one ? L::kOneSlots : L::kChunkSlots;
      const uint32_t abase = one ? L::kSumCol : L::kSumCol + BN;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        for (int c = 0; c < nch && ok; ++c, ++cseq) {
          const int b = cseq & 1;
          if (!mbar_wait_bounded(&accempty[b], ((cseq >> 1) & 1) ^ 1)) {
            report_error(err, kErrTimeoutMma);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + b * BN;
          const int kb1 = (c + 1) * chunk_kb < nkb ? (c + 1) * chunk_kb : nkb;
          for (int kb = c * chunk_kb; kb < kb1; ++kb) {
            // The converters wait for the stage's copies before they arrive on afull, so this wait
            // also orders the x tile (one wait per stage instead of two: 372 -> 354 us at M = 4096,
            // N = 11008)
            if (!mbar_wait_bounded(&afull[aslot], aph)) {
              report_error(err, kErrTimeoutMma);
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t xs_s = smem_u32(smem + stage * L::kStage);
            const uint32_t a_tmem = tmem_base + abase + aslot * 64;
            // the stage's B descriptors differ only in the start address field (bits 0-13, addr >> 4;
            // shared-memory addresses stay below 2^18, so adding to it never carries)
            const uint64_t bdesc0 = umma_sdesc_sw128(xs_s, 16, 1024);
#pragma unroll
            for (int s = 0; s < kBK / 16; ++s) {
              // k16 step s: x box s / 4, 32 bytes per step along its 128-byte rows
              const uint64_t bdesc = bdesc0 + (uint64_t)(((s >> 2) * L::kXBox + (s & 3) * 32) >> 4);
              umma_f16_ta(d_tmem, a_tmem + s * 8, bdesc, idesc, (kb > c * chunk_kb || s > 0) ? 1u : 0u);
            }
            umma_commit(&empty[stage]);  // the stage and this block's A slot are free again
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
            if (++aslot == nslots) {
              aslot = 0;
              aph ^= 1;
            }
          }
          if (!ok) break;
          umma_commit(&accfull[b]);
        }
      }
      umma_commit(finalbar);
      if (!mbar_wait_bounded(finalbar, 0)) report_error(err, kErrTimeoutDrain);
    }
  } else if (warp < kEpiWarp0) {
    // ---------------- converters: int8 weight tile -> fp16 A operand in TMEM ----------------
    const int quad = warp & 3;                // TMEM lane quadrant this warp may access
    const int half = (warp - kCvWarp0) >> 2;  // k half of the tile: bytes [64 half, 64 half + 64)
    const int row = quad * 32 + lane;         // output channel within the tile = TMEM lane
    const int sw = row & 7;                   // 128-byte swizzle: 16-byte chunk c sits at c ^ sw
    int stage = 0, phase = 0, aslot = 0, kbi = 0;
    bool ok = mbar_wait_warp(modebar, 0);
    if (!ok) report_error(err, kErrTimeoutFull);
    const bool one = ok && mode_smem[1] != 0;
    const int nslots = one ? L::kOneSlots : L::kChunkSlots;
    const uint32_t lane_addr =
        tmem_base + ((uint32_t)(quad * 32) << 16) + (one ? L::kSumCol : L::kSumCol + BN) + 32 * half;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      for (int kb = 0; kb < nkb; ++kb, ++kbi) {
        // the A slot was last used by block kbi - nslots: wait until its MMAs have completed
        const int prev = kbi - nslots;
        const bool okf = mbar_wait_warp(&full[stage], phase);
        const bool oke = prev < 0 || mbar_wait_warp(&empty[prev % kStages], (prev / kStages) & 1);
        if (!okf || !oke) {
          report_error(err, kErrTimeoutFull);
          ok = false;
          break;
        }
        const uint32_t wrow = smem_u32(smem + stage * L::kStage + L::kOffW) + row * kBK;
        uint32_t a[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = lds_u128(wrow + (((4 * half + c) ^ sw) << 4));
          i8x4_to_f16x2x2(v.x, a[8 * c + 0], a[8 * c + 1]);
          i8x4_to_f16x2x2(v.y, a[8 * c + 2], a[8 * c + 3]);
          i8x4_to_f16x2x2(v.z, a[8 * c + 4], a[8 * c + 5]);
          i8x4_to_f16x2x2(v.w, a[8 * c + 6], a[8 * c + 7]);
        }
        tmem_st_32x32b_x32(lane_addr + aslot * 64, a);
        tmem_st_wait();
        tc_fence_before_sync();
        // the int8 tile was read through the generic proxy; its TMA refill (async proxy) follows this
        // release, and only a proxy fence orders the two
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[aslot]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++aslot == nslots) aslot = 0;
      }
    }
  } else {
    // ---------------- epilogue: exact int32 from the chunk accumulators ----------------
    const int ew = warp - kEpiWarp0;
    const int quad = warp & 3;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    const uint32_t sum_col = L::kSumCol;
    // The accumulation mode, for the whole launch: one exact chunk when 128 x every row's L1 norm
    // stays within 2^24.  These warps reduce the pre-pass blocks' maxima and publish the mode
    // (modebar) to the MMA thread and the converters, which wait for it before their first stage.
    int mx = 0;
    if (blockmax)
      for (int b = (warp - kEpiWarp0) * 32 + lane; b < nbm; b += kEpiWarps * 32) mx = max(mx, __ldg(blockmax + b));
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) atomicMax(&mode_smem[0], mx);
    named_barrier_sync(1, kEpiWarps * 32);
    const bool one = blockmax != nullptr && mode_smem[0] <= kOneChunkL1;
    if (warp == kEpiWarp0 && lane == 0) {
      mode_smem[1] = one ? 1 : 0;
      mbar_arrive(modebar);
    }
    const int nch = one ? 1 : nchunks;
    BoxStage<L::kBufs> out;
    out.init(reinterpret_cast<__half*>(smem + L::kOffOut + ew * L::kBufs * L::kBox), rfull + ew * L::kBufs, &tm_y,
             &tm_r, ea.residual != nullptr);
    int cseq = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const int nt = tile % ntn, mt = tile / ntn;
      const int n0 = nt * kBM + quad * 32, n = n0 + lane;
      const float wn = n < N ? ws[n] : 0.f;
      const float bn = (ea.bias && n < N) ? __half2float(ea.bias[n]) : 0.f;
      for (int c = 0; c < nch && ok; ++c, ++cseq) {
        const int b = cseq & 1;
        const bool first = c == 0, last = c == nch - 1;
        if (last) out.begin(n0, mt * BN, BN / 32, lane);  // residual boxes land while the last chunk's MMAs run
        if (!mbar_wait_warp(&accfull[b], (cseq >> 1) & 1)) {
          report_error(err, kErrTimeoutMma);
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j) {
          uint32_t r[32], sacc[32];
          tmem_ld_32x32b_x32(lane_base + b * BN + 32 * j, r);
          if (!first) tmem_ld_32x32b_x32(lane_base + sum_col + 32 * j, sacc);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int v = __float2int_rn(__uint_as_float(r[k]));  // an exact integer below 2^24
            sacc[k] = first ? (uint32_t)v : (uint32_t)((int)sacc[k] + v);
          }
          if (!last) {
            tmem_st_32x32b_x32(lane_base + sum_col + 32 * j, sacc);
            tmem_st_wait();
            continue;
          }
          const int mbase = mt * BN + 32 * j;
          const float xl = mbase + lane < M ? xs[mbase + lane] : 0.f;
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
            const int a = (int)sacc[k];
            const float rr = out.has_res ? __half2float(bx[k * 32 + lane]) : 0.f;
            bx[k * 32 + lane] = __float2half_rn(add_terms(__fmul_rn(__fmul_rn(__int2float_rn(a), xm), wn), ea, bn, rr));
            if (acc_out && n < N && mbase + k < M) acc_out[(size_t)(mbase + k) * N + n] = a;
          }
          out.store(j, bx, lane);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[b]);
      }
    }
    if (!out.finish(lane)) report_error(err, kErrTimeoutDrain);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, L::kTmemCols);
}

template <int BN>
cudaError_t launch_q(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, const CUtensorMap& tr,
                     const float* xs, const float* ws, int M, int N, int K, int32_t* acc_out, EpilogueAdd ea,
                     const int* blockmax, int nbm, unsigned* dev_err, cudaStream_t stream) {
  using L = QLayout<BN>;
  auto kern = w8a8_prefill_kernel<BN>;
  static std::atomic<bool> attr_set[64];  // per device; racing first calls set the same attribute
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const int ntiles = ((N + kBM - 1) / kBM) * ((M + BN - 1) / BN);
  const int grid = ntiles < num_sms() ? ntiles : num_sms();
  kern<<<grid, kThreads, L::kBytes, stream>>>(tx, tw, xs, ws, M, N, K, ty, tr, acc_out, ea, blockmax, nbm, dev_err);
  return cudaGetLastError();
}

}  // namespace

// [M][K] fp16 copy of the codes, then the pre-pass blocks' largest row L1 norms (int32)
size_t w8a8_prefill_workspace_bytes(int M, int K) { return (size_t)M * (size_t)K * 2 + kPrepassMaxBlocks * 4; }

cudaError_t launch_w8a8_prefill(const int8_t* q, const float* xs, const int8_t* qw, const float* ws, int M, int K,
                                int N, uint16_t* y, int32_t* acc_out, const uint16_t* bias, const uint16_t* residual,
                                void* workspace, unsigned* dev_err, cudaStream_t stream, std::string* err) {
  const EpilogueAdd ea{reinterpret_cast<const __half*>(bias), reinterpret_cast<const __half*>(residual)};
  // 1. activation codes -> exact fp16 in the workspace, and the blocks' largest row L1 norms after them
  __half* xh = reinterpret_cast<__half*>(workspace);
  int* blockmax = reinterpret_cast<int*>(reinterpret_cast<char*>(workspace) + (size_t)M * K * 2);
  long long blocks = ((long long)M + 7) / 8;  // eight rows (warps) per block
  if (blocks > 4L * num_sms()) blocks = 4L * num_sms();
  if (blocks > kPrepassMaxBlocks) blocks = kPrepassMaxBlocks;
  const int grid = (int)blocks;
  i8_to_f16_rows_kernel<<<grid, 256, 0, stream>>>(q, xh, blockmax, M, K);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // 2. the GEMM
  const int BN = M <= 64 ? 64 : 128;
  CUtensorMap tx, tw, ty, tr;
  if (!make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xh, K, M, (uint64_t)K * 2, 64, BN,
                    CU_TENSOR_MAP_SWIZZLE_128B, err) ||
      !make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qw, K, N, (uint64_t)K, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B,
                    err) ||
      !make_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, y, N, M, (uint64_t)N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE,
                    err) ||
      (residual && !make_tmap_2d(&tr, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, residual, N, M, (uint64_t)N * 2, 32, 32,
                                 CU_TENSOR_MAP_SWIZZLE_NONE, err))) {
    return cudaErrorInvalidValue;
  }
  if (!residual) tr = ty;  // not read
  if (BN == 64) return launch_q<64>(tx, tw, ty, tr, xs, ws, M, N, K, acc_out, ea, blockmax, grid, dev_err, stream);
  return launch_q<128>(tx, tw, ty, tr, xs, ws, M, N, K, acc_out, ea, blockmax, grid, dev_err, stream);
}

}  // namespace wql
