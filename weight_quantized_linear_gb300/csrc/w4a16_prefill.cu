// w4a16_prefill.cu -- AWQ W4A16 GEMM for prefill-shaped calls on the tcgen05 tensor cores.
//
// y[m, n] = sum_k x[m, k] * (q[k, n] - z[k/G, n]) * s[k/G, n] ("LMDeploy ... INT4 quantisation"
// tutorial, section 2; section 5.1 names the engine's fp16 x int4 GEMM).  Tiles of 128 output
// channels x BN tokens (BN = 32, 64, 128, 192 or 256), K walked in blocks of 128, one ring of stages
// [x tile | packed | s | z]:
//   * warps 0 and 14, one thread each: TMA copies of the packed weight tile with its scale /
//     zero-point rows, and of the activation tile (K-major, 128B swizzle);
//   * warps 2-9: dequantise the packed tile into the MMA's A operand, fp16 (q - z) * s (exact q - z
//     via the 1024 + q bit-splice trick, one rounding for the scale), written to tensor memory
//     with tcgen05.st, one channel per TMEM lane, so that shared memory carries only the
//     activations and the packed weights;
//   * warp 1: allocates TMEM; one thread issues tcgen05.mma.kind::f16 (M = 128 channels,
//     N = BN tokens, K = 16, A from TMEM) into an fp32 accumulator and commits stage releases.
//     BN <= 128: two accumulators, so a tile's epilogue overlaps the next tile's MMAs; BN = 192 and
//     256: one accumulator (512 TMEM columns hold it and the A slots) and a three-stage ring, the
//     larger MMAs carrying more work per issued instruction than the 128-token tile's;
//   * warps 10-13: tcgen05.ld the accumulator (lane = channel, column = token), round to fp16, store.
// Swapping A and B puts the dequantised weights (not the activations) in the 128-row operand, so
// the dequantisers write 128 x kBK fp16 per stage whatever the token count.
//
// Two launch shapes:
//   * persistent (gridDim.y == 1): one CTA per SM walks the tiles;
//   * split-K (gridDim.y == S in {2, 4, 8}, clusters of S CTAs along y): when the tiles are fewer
//     than half the SMs, the S CTAs of a cluster each take 1/S of K for one tile.  After their
//     main loops they exchange partial sums through distributed shared memory by bulk copies
//     (send buffers in the stage ring; receive buffers in the ring, or in shared memory of their
//     own for 32- and 64-token tiles): CTA r owns token columns [r BN/S, (r+1) BN/S) and every
//     warp then adds the S partials in split order, so the result does not depend on timing.
// Launched with programmatic dependent launch: the packed weights of the first stages are
// requested before waiting for the preceding kernel, whose output may be x.
#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "trace.cuh"

namespace wql {
namespace {

constexpr int kBK = 128;         // k per stage: eight MMAs per barrier round trip of the MMA thread
constexpr int kBM = 128;         // output channels per tile (MMA M)
constexpr int kStripWords = 16;  // packed words per tile row
// Warp 0 issues the weight copies and warp 14 the activation copies: copies issued by one thread
// complete one after another, so two issuing warps keep twice as many in progress.
constexpr int kProducerWarp = 0, kMmaWarp = 1, kDqWarp0 = 2, kDqWarps = 8, kEpiWarp0 = 10, kEpiWarps = 4;
constexpr int kXProducerWarp = kEpiWarp0 + kEpiWarps;
constexpr int kThreads = (kXProducerWarp + 1) * 32;

constexpr int imin(int a, int b) { return a < b ? a : b; }

// NACC accumulators in TMEM: 2 when a CTA walks several tiles (a tile's epilogue then overlaps the
// next tile's MMAs), 1 when it owns one tile, which leaves TMEM for more A slots and so a deeper
// ring.  Each stage owns one 64-column A slot, so the ring depth is the smaller of what shared
// memory and TMEM hold (at most 8).  The pipeline of the smaller tiles is latency-bound: a stage's
// copy, its dequantisation and its MMAs follow one another before the stage is refilled (128-token
// tiles, one tile per CTA: 4 -> 5 stages).
template <int BN, int LG, int NACC>
struct PLayout {
  static_assert(NACC == 1 || (NACC == 2 && BN <= 128), "192- and 256-token tiles have one accumulator");
  static constexpr int G = 1 << LG;
  static constexpr int kGR = G >= kBK ? 1 : kBK / G;
  static constexpr int kXBox = BN * 128;                 // BN token rows x 64 k fp16
  static constexpr int kXBoxes = kBK / 64;
  static constexpr int kXBytes = kXBoxes * kXBox;
  static constexpr int kWBytes = kBK * kStripWords * 4;  // kBK rows x 16 packed words
  static constexpr int kSBytes = kGR * kBM * 2;
  static constexpr int kZBytes = kGR * kStripWords * 4;
  static constexpr int kOffW = kXBytes;                  // 1024-aligned (the packed tile needs 512)
  static constexpr int kOffS = kOffW + kWBytes;
  static constexpr int kOffZ = kOffS + kSBytes;
  static constexpr int kStage = (kOffZ + kZBytes + 1023) / 1024 * 1024;
  // stage s also owns TMEM A slot s: the producers' wait for the stage to be free (the MMAs of the
  // stage kStages earlier have completed) frees the slot too
  static constexpr int kAccBufs = NACC;
  static constexpr int kMaxBarBytes = (3 * 8 + 6) * 8 + 16;
  // 32- and 64-token tiles keep a split-K receive buffer of their own after the barriers, sized for
  // the largest split (S = 8: kBM x (BN / 8 + 4) fp32 from each of 8 splits), without costing a
  // ring stage: peers may then send before this CTA's main loop is over.  Larger tiles receive
  // into their ring once every main loop of the cluster is over.
  static constexpr bool kOwnRecv = BN <= 64;
  static constexpr int kRecvBytes = kOwnRecv ? kBM * (BN + 4 * 8) * 4 : 0;
  static constexpr int kStages =
      imin(8, imin((227 * 1024 - 1024 - kMaxBarBytes - kRecvBytes) / kStage, (512 - NACC * BN) / 64));
  static constexpr uint32_t kWTx = kWBytes + kSBytes + kZBytes;
  static constexpr int kBarBytes = (3 * kStages + 6) * 8 + 16;
  static constexpr int kOffRecv = (kStages * kStage + kBarBytes + 127) / 128 * 128;
  static constexpr int kBytes = kOffRecv + kRecvBytes + 1024;
  static constexpr uint32_t kAColBase = kAccBufs * BN;  // A slots (64 columns = 128 k each) after the accumulators
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kAColBase + 64 * kStages <= kTmemCols, "TMEM budget");
  // split-K exchange buffers (alias the ring once every main loop of the cluster has ended): a
  // receive buffer [source split][channel][BN / S + 4] fp32 and a send buffer with the same chunks
  // for the S - 1 other owners: 2 S - 1 chunks of kBM (BN / S + 4) fp32
  static constexpr int exchange_bytes(int S) { return (2 * S - 1) * kBM * (BN / S + 4) * 4; }
  static constexpr bool split_fits(int S) {
    return S == 1 || (BN / S >= 4 && (kOwnRecv ? S <= 8 && (S - 1) * kBM * (BN / S + 4) * 4 <= kStages * kStage
                                               : exchange_bytes(S) <= kStages * kStage));
  }
  static_assert(split_fits(2), "a two-way split must fit");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// The output channel (within the 128-channel tile) held by TMEM lane i: the dequantisers' stores put
// channel 32 q + 4 g + e (g = 0..7, e = 0..3) in lane 32 q + 8 e + g.
__device__ __forceinline__ int tmem_lane_channel(int i) { return 32 * (i >> 5) + 4 * (i & 7) + ((i >> 3) & 3); }

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

// Every thread of every warp calls this the same number of times (cluster barrier, release/acquire).
__device__ __forceinline__ void cluster_phase() {
  __syncwarp();
  cluster_arrive_release();
  cluster_wait();
}

template <int BN, int LG, int NACC>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_prefill_kernel(const __grid_constant__ CUtensorMap tm_x,   // x [M][K] fp16, box {64, BN}, SW128
                         const __grid_constant__ CUtensorMap tm_qw,  // qweight [K][N/8]: box {16, 64}, or (A in TMEM)
                                                                     // 3D {N/8, K/4, 4} box {16, 32, 4}, SW64
                         const __grid_constant__ CUtensorMap tm_s,   // scales [K/G][N], box {128, GR}
                         const __grid_constant__ CUtensorMap tm_z,   // qzeros [K/G][N/8], box {16, GR}
                         int M, int N, int K, __half* __restrict__ y, int act, unsigned* err) {
  using L = PLayout<BN, LG, NACC>;
  constexpr int kStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * L::kStage);
  uint64_t* empty = full + kStages;
  uint64_t* afull = empty + kStages;
  uint64_t* accfull = afull + kStages;  // [2]
  uint64_t* accempty = accfull + 2;     // [2]
  uint64_t* finalbar = accempty + 2;    // [1]
  uint64_t* recvbar = finalbar + 1;     // [1] split-K: this CTA's receive buffer is complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(recvbar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntn = (N + kBM - 1) / kBM;
  const int ntm = (M + BN - 1) / BN;
  const int ntiles = ntn * ntm;
  const int nkb = (K + kBK - 1) / kBK;
  // phase stamps (trace builds only): 0 start, 1 TMEM allocated, 2 dependency resolved, 3 first
  // stage's MMAs may start, 4 last stage's MMAs may start, 5 last MMAs issued, 6 accumulator ready
  // (first tile), 7 split-K cluster barrier passed, 8 partials sent, 9 partials received,
  // 10 outputs stored, 11 end; the ninth stage of the first tile: 12 at the dequantisers (first
  // warp), 13 dequantised, 14 at the MMA thread, 15 its MMAs issued
  WQL_TRACE_ROW(y);
  if (threadIdx.x == 0) {
    WQL_STAMP(0);
    WQL_STAMP_SMID();
  }
  const int S = gridDim.y, split = blockIdx.y;  // split-K: cluster (1, S, 1), rank = blockIdx.y
  const int kb0 = (int)(((long long)split * nkb) / S), kb1 = (int)(((long long)(split + 1) * nkb) / S);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 2);               // the weight and the activation producer
      mbar_init(&empty[s], 1);              // tcgen05.commit of the MMAs reading the stage
      mbar_init(&afull[s], kDqWarps);       // one arrival per dequantising warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], kEpiWarps);
    }
    mbar_init(finalbar, 1);
    mbar_init(recvbar, 1);
    fence_mbarrier_init();
    // split-K: every other CTA of the cluster sends this CTA its partials of the token columns it
    // owns, one bulk copy of kBM x (BN / S + 4) fp32 each
    if (gridDim.y > 1)
      mbar_arrive_expect_tx(recvbar, (uint32_t)((gridDim.y - 1) * kBM * (BN / gridDim.y + 4) * 4));
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // split-K with a receive buffer of its own: cluster phase 0 (arrive now, wait before the first
  // copy to a peer) guarantees every peer's receive barrier is initialised
  if (L::kOwnRecv && gridDim.y > 1) cluster_arrive_relaxed();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) WQL_STAMP(1);
  // A grid of at most one tile per CTA leaves SMs free for most of its run: let the next kernel be
  // scheduled on them now and start its own weight prefetch (its consumers still wait for this
  // grid to complete).  A persistent grid over many tiles triggers only when it exits.
  if (threadIdx.x == 0 && ntiles <= (int)gridDim.x) grid_dependents_launch();

  // One tile per CTA (every split-K launch, and grids with no more tiles than CTAs): once the
  // accumulator is ready the dequantisers are idle, so they drain it together with the epilogue
  // warps.  Each TMEM lane quarter has three such warps, and the quarter's 32-column chunk j goes to
  // drain rank j % 3 (0: its epilogue warp, 1 and 2: its two dequantisers).  CTAs that walk several
  // tiles drain with the four epilogue warps alone while the dequantisers move on to the next tile.
  const bool single = ntiles <= (int)gridDim.x;
  constexpr int kDrainRanks = 3, kDrainWarps = kEpiWarps + kDqWarps;
  auto drain_single = [&](int quad, int rank) {
    const int i = quad * 32 + lane;
    // channel of TMEM lane i: lane 32 q + L holds channel 32 q + 4 (L % 8) + L / 8
    const int col_in_tile = tmem_lane_channel(i);
    const int pair_mask = 8;  // gate/up pairs meet in lanes differing in bit 3 (see the epilogue)
    const int NO = act ? N / 2 : N;
    const int nt = (int)blockIdx.x % ntn, mt = (int)blockIdx.x / ntn;
    const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16);
    const bool ready = mbar_wait_warp(&accfull[0], 0);
    if (!ready) report_error(err, kErrTimeoutMma);
    tc_fence_after_sync();
    if (threadIdx.x == kEpiWarp0 * 32) WQL_STAMP(6);
    if (S == 1) {
      grid_dependency_wait();  // y may still be read by the preceding kernel
      const int n = nt * kBM + col_in_tile;
#pragma unroll 1
      for (int cc = 32 * rank; ready && cc < BN; cc += 32 * kDrainRanks) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + cc, r);
        tmem_ld_wait();
        const int mbase = mt * BN + cc;
        if (act) {
          const bool even = (n & 1) == 0;
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float v0 = __uint_as_float(r[k]), v1 = __uint_as_float(r[k + 1]);
            const float got = __shfl_xor_sync(0xffffffffu, even ? v1 : v0, pair_mask);
            const int m = mbase + k + (even ? 0 : 1);
            const __half o = silu_mul_h(even ? v0 : got, even ? got : v1);  // (gate, up)
            if (n < N && m < M) y[(size_t)m * NO + n / 2] = o;
          }
        } else if (n < N) {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            if (mbase + k < M) y[(size_t)(mbase + k) * N + n] = __float2half_rn(__uint_as_float(r[k]));
          }
        }
      }
      return;
    }
    // split-K: exactly one tile per cluster (the host launches gridDim.x == ntiles)
    const int CW = BN / S;       // token columns owned by each CTA of the cluster
    const int rstride = CW + 4;  // floats per exchange row (16 bytes of padding against bank conflicts)
    const uint32_t chunk = (uint32_t)(kBM * rstride * 4);
    if constexpr (L::kOwnRecv)
      cluster_wait();    // (0) every peer is initialised; its own receive buffer is always free
    else
      cluster_phase();   // (1) every main loop of the cluster is over: the rings are free
    if (threadIdx.x == kEpiWarp0 * 32) WQL_STAMP(7);
    // recv [S][kBM][rstride]: the partials of this CTA's columns, its own written here directly;
    // sendb [S - 1][kBM][rstride]: this CTA's partials of the other owners' columns (in the ring,
    // which this CTA's own main loop no longer uses)
    const uint32_t recv = L::kOwnRecv ? smem_u32(smem + L::kOffRecv) : smem_u32(smem);
    const uint32_t sendb = L::kOwnRecv ? smem_u32(smem) : recv + (uint32_t)S * chunk;
    // With owner ranges of at most 32 columns, the rows of this warp's lane quarter in each owner's
    // chunk are written by this warp alone: it sends them as soon as they are staged, one bulk copy
    // per (lane quarter, owner), so the copies overlap the staging and come from up to twelve
    // warps.  Wider owner ranges span several warps' chunks: one thread sends whole chunks after a
    // barrier of the draining warps.
    const bool per_warp = CW <= 32;
    const uint32_t rbar = smem_u32(recvbar);
    const uint32_t qoff = (uint32_t)(32 * quad * rstride * 4), qbytes = (uint32_t)(32 * rstride * 4);
#pragma unroll 1
    for (int cc = 32 * rank; cc < BN; cc += 32 * kDrainRanks) {
      uint32_t r[32];
      if (ready) {
        tmem_ld_32x32b_x32(taddr + cc, r);
        tmem_ld_wait();
      } else {  // the accumulator never became ready (an error is reported): send zeros, so that
                // the peers' receive barriers still complete
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = 0u;
      }
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const int col = cc + 4 * g;
        const int owner = col / CW, cl = col - owner * CW;
        const uint32_t base = owner == split ? recv + (uint32_t)split * chunk
                                             : sendb + (uint32_t)(owner < split ? owner : owner - 1) * chunk;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + (uint32_t)((i * rstride + cl) * 4)),
                     "r"(r[4 * g]), "r"(r[4 * g + 1]), "r"(r[4 * g + 2]), "r"(r[4 * g + 3])
                     : "memory");
      }
      if (per_warp) {
        fence_proxy_async_smem();  // the staged rows are read by the bulk copies (async proxy)
        __syncwarp();
        if (lane == 0) {
          for (int o = cc / CW; o <= (cc + 31) / CW; ++o) {
            if (o == split) continue;
            bulk_copy_to_peer(map_cluster_addr(recv + (uint32_t)split * chunk + qoff, (uint32_t)o),
                              sendb + (uint32_t)(o < split ? o : o - 1) * chunk + qoff, qbytes,
                              map_cluster_addr(rbar, (uint32_t)o));
          }
        }
      }
    }
    tc_fence_before_sync();
    if (!per_warp) {
      fence_proxy_async_smem();  // the send chunks are read by the bulk copies (async proxy)
      named_barrier_sync(1, kDrainWarps * 32);
      // One bulk copy per other owner, into its receive slot `split`: the copy engine moves the
      // chunks (st.shared::cluster or st.async stores from the epilogue threads took 3-10 us for a
      // 128 x 128 tile).
      if (threadIdx.x == kEpiWarp0 * 32) {
        for (int o = 0; o < S; ++o) {
          if (o == split) continue;
          bulk_copy_to_peer(map_cluster_addr(recv + (uint32_t)split * chunk, (uint32_t)o),
                            sendb + (uint32_t)(o < split ? o : o - 1) * chunk, chunk,
                            map_cluster_addr(rbar, (uint32_t)o));
        }
      }
    }
    if (threadIdx.x == kEpiWarp0 * 32) WQL_STAMP(8);
    // every other CTA's chunk has landed once the receive barrier completes
    if (rank == 0) {
      if (!mbar_wait_warp(recvbar, 0)) report_error(err, kErrTimeoutMma);
      if (threadIdx.x == kEpiWarp0 * 32) WQL_STAMP(9);
    }
  };

  if (warp == kProducerWarp || warp == kXProducerWarp) {
    // ---------------- producers: weights (warp 0) and activations (warp 14) ----------------
    if (lane == 0) {
      const bool wprod = warp == kProducerWarp;
      if (wprod) {
        tma_prefetch_desc(&tm_qw);
        tma_prefetch_desc(&tm_s);
        tma_prefetch_desc(&tm_z);
      } else {
        tma_prefetch_desc(&tm_x);
        grid_dependency_wait();  // the activations may come from the preceding kernel
        WQL_STAMP(2);
      }
      // The packed weights do not depend on the preceding kernel: the weight producer never waits
      // for it, so its first stages stream while the preceding kernel is still running.
      int stage = 0, phase = 0, issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const int nt = tile % ntn, mt = tile / ntn;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1)) {
            report_error(err, kErrTimeoutEmpty);
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * L::kStage;
          if (wprod) {
            mbar_arrive_expect_tx(&full[stage], L::kWTx);
            // rows k = 4a + b land at row 32 b + a of the tile
            tma_load_3d(st + L::kOffW, &tm_qw, &full[stage], nt * kStripWords, kb * (kBK / 4), 0);
            tma_load_2d(st + L::kOffS, &tm_s, &full[stage], nt * kBM, (kb * kBK) >> LG);
            tma_load_2d(st + L::kOffZ, &tm_z, &full[stage], nt * kStripWords, (kb * kBK) >> LG);
          } else {
            mbar_arrive_expect_tx(&full[stage], L::kXBytes);
#pragma unroll
            for (int b = 0; b < L::kXBoxes; ++b)
              tma_load_2d(st + b * L::kXBox, &tm_x, &full[stage], kb * kBK + 64 * b, mt * BN);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: wait for the copies of the last (up to kStages) issued stages.
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
      constexpr uint32_t idesc = umma_idesc_f16(kBM, BN, /*A from TMEM*/ 0, /*B K-major*/ 0);
      int stage = 0, phase = 0, it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++it) {
        const int b = it % L::kAccBufs;
        if (!mbar_wait_bounded(&accempty[b], ((it / L::kAccBufs) & 1) ^ 1)) {
          report_error(err, kErrTimeoutMma);
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + b * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          // The dequantisers wait for the stage's copies before they arrive on afull, so that wait
          // also orders the x tile (one wait per stage: M = 64, N = 12288: 19.0 -> 18.0 us)
          if (!mbar_wait_bounded(&afull[stage], phase)) {
            report_error(err, kErrTimeoutMma);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (kb == kb0 && it == 0) WQL_STAMP(3);
          if (kb == kb1 - 1) WQL_STAMP(4);
          if (kb == kb0 + 8 && it == 0) WQL_STAMP(14);
          const uint32_t xs = smem_u32(smem + stage * L::kStage);
          // the B descriptors of the stage differ only in the start address (bits 0-13, addr >> 4;
          // shared-memory addresses stay below 2^18, so adding to it never carries)
          const uint64_t bdesc0 = umma_sdesc_sw128(xs, 16, 1024);
#pragma unroll
          for (int s = 0; s < kBK / 16; ++s) {
            // B: 64-k boxes of K-major 128-byte rows, 8-row groups 1 KB apart; a k16 step is 32
            // bytes along the row.  A: TMEM slot `stage`, eight columns per k16 step.
            const uint64_t bdesc = bdesc0 + (uint64_t)(((s >> 2) * L::kXBox + (s & 3) * 32) >> 4);
            const uint32_t acc = (kb != kb0 || s != 0) ? 1u : 0u;
            umma_f16_ta(d_tmem, tmem_base + L::kAColBase + stage * 64 + s * 8, bdesc, idesc, acc);
          }
          if (kb == kb0 + 8 && it == 0) WQL_STAMP(15);
          umma_commit(&empty[stage]);  // the stage is free once these MMAs have read it
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        WQL_STAMP(5);
        umma_commit(&accfull[b]);
      }
      // every MMA issued by this thread has completed before TMEM is released
      umma_commit(finalbar);
      if (!mbar_wait_bounded(finalbar, 0)) report_error(err, kErrTimeoutDrain);
    }
  } else if (warp < kEpiWarp0) {
    // ---------------- dequantisers: packed int4 -> fp16 A operand in TMEM ----------------
    // Warp w writes TMEM lane quarter q = w % 4 (channels 32 q ..) for k in [64 hk, 64 hk + 64) of
    // each stage.  Thread (g, c) = (lane / 4, lane % 4) takes packed word 4 q + g / 2, nibbles
    // 4 (g % 2) + e (e = 0..3), i.e. channels 32 q + 4 g + e, at k = 16 m + 4 c + {0..3}; through
    // tcgen05.st.16x256b, e = 0, 1 go to lanes g, g + 8 and e = 2, 3 to lanes 16 + g, 24 + g, so
    // TMEM lane 32 q + L holds channel 32 q + 4 (L % 8) + L / 8.  Rows k and k + 1 are paired by
    // one PRMT, so each 32-bit value is the fp16 pair (k, k + 1) of one channel: a TMEM column.
    const int dw = warp - kDqWarp0;
    const int q = warp & 3, hk = dw >> 2;
    const int g = lane >> 2, c = lane & 3;
    const int wj = 4 * q + (g >> 1);
    const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
    const uint32_t taddr0 = tmem_base + ((uint32_t)(32 * q) << 16) + L::kAColBase + 32 * hk;
    const uint32_t taddr1 = taddr0 + (16u << 16);
    constexpr uint32_t kMagic = 0x64006400u, kSixteenth = 0x2C002C00u;
    int stage = 0, phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_warp(&full[stage], phase)) {  // warp-uniform: tcgen05.st is .sync.aligned
          report_error(err, kErrTimeoutFull);
          ok = false;
          break;
        }
        tc_fence_after_sync();  // this slot's earlier MMAs (ordered through the stage barriers) come first
        if (threadIdx.x == kDqWarp0 * 32 && kb == kb0 + 8 && tile == (int)blockIdx.x) WQL_STAMP(12);
        const uint32_t st = smem_u32(smem + stage * L::kStage);
        uint32_t r0[16], r1[16];
        uint32_t zc[4], sp[4];  // per channel e: -(1024 + z) or -(64 + z), and s, in both halves
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          // the quantisation group changes within the warp's 64 k only when G = 32 (at m = 2)
          if (m == 0 || (L::kGR == 4 && m == 2)) {
            const int gi = L::kGR == 1 ? 0 : ((64 * hk + 16 * m) >> LG);
            const uint32_t zw = lds_u32(st + L::kOffZ + gi * (kStripWords * 4) + wj * 4) >> (16 * (g & 1));
            uint32_t sv0, sv1;  // scales of channels 32 q + 4 g + {0, 1} and {2, 3}
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                         : "=r"(sv0), "=r"(sv1)
                         : "r"(st + L::kOffS + gi * (kBM * 2) + (32 * q + 4 * g) * 2));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t v = (zw >> (4 * e)) & 15u;
              // codes spliced as 1024 + q take -(1024 + z); codes spliced as 1024 + 16 q, scaled by
              // 1/16, take -(64 + z)
              zc[e] = (e & 1) ? (0xD400D400u | (v << 4) | (v << 20)) : (0xE400E400u | v | (v << 16));
              const uint32_t sw = e < 2 ? sv0 : sv1;
              sp[e] = prmt(sw, sw, (e & 1) ? 0x3232u : 0x1010u);
            }
          }
          uint32_t w[4];
#pragma unroll
          for (int dd = 0; dd < 4; ++dd) {
            // k = 64 hk + 16 m + 4 c + dd sits at tile row 32 dd + 16 hk + 4 m + c (64-byte rows,
            // 16-byte chunk index XOR bits 1-2 of the row)
            const int row = 32 * dd + 16 * hk + 4 * m + c;
            w[dd] = lds_u32(st + L::kOffW + row * 64 + ((q ^ ((row >> 1) & 3)) << 4) + (g >> 1) * 4);
          }
          const uint32_t t01 = prmt(w[0], w[1], sel), t23 = prmt(w[2], w[3], sel);
          const uint32_t t01h = t01 >> 8, t23h = t23 >> 8;
          // channel e of the pair (k, k + 1) from t01 (column 8 m + 2 c) and (k + 2, k + 3) from t23
          r0[4 * m + 0] = hmul2_u32(hadd2_u32(and_or(t01, 0x000F000Fu, kMagic), zc[0]), sp[0]);
          r0[4 * m + 1] = hmul2_u32(hadd2_u32(and_or(t23, 0x000F000Fu, kMagic), zc[0]), sp[0]);
          r0[4 * m + 2] = hmul2_u32(hfma2_u32(and_or(t01, 0x00F000F0u, kMagic), kSixteenth, zc[1]), sp[1]);
          r0[4 * m + 3] = hmul2_u32(hfma2_u32(and_or(t23, 0x00F000F0u, kMagic), kSixteenth, zc[1]), sp[1]);
          r1[4 * m + 0] = hmul2_u32(hadd2_u32(and_or(t01h, 0x000F000Fu, kMagic), zc[2]), sp[2]);
          r1[4 * m + 1] = hmul2_u32(hadd2_u32(and_or(t23h, 0x000F000Fu, kMagic), zc[2]), sp[2]);
          r1[4 * m + 2] = hmul2_u32(hfma2_u32(and_or(t01h, 0x00F000F0u, kMagic), kSixteenth, zc[3]), sp[3]);
          r1[4 * m + 3] = hmul2_u32(hfma2_u32(and_or(t23h, 0x00F000F0u, kMagic), kSixteenth, zc[3]), sp[3]);
        }
        tmem_st_16x256b_x4(taddr0 + stage * 64, r0);
        tmem_st_16x256b_x4(taddr1 + stage * 64, r1);
        tmem_st_wait();
        tc_fence_before_sync();  // the stores are ordered before the MMA thread's wait on afull
        // the packed tile was read through the generic proxy; its TMA refill (async proxy) follows
        // this release, and only a proxy fence orders the two
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[stage]);
        if (threadIdx.x == kDqWarp0 * 32 && kb == kb0 + 8 && tile == (int)blockIdx.x) WQL_STAMP(13);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (single) drain_single(q, 1 + hk);
  } else if (warp < kEpiWarp0 + kEpiWarps) {
    // ---------------- epilogue: TMEM -> fp16 -> global ----------------
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    if (single) {
      drain_single(quad, 0);
    } else {
      // several tiles per CTA (never split-K): accumulators b = it % 2 alternate
      const int i = quad * 32 + lane;
      // channel of TMEM lane i: lane 32 q + L holds channel 32 q + 4 (L % 8) + L / 8
      const int col_in_tile = tmem_lane_channel(i);
      // with the gate/up activation (act), channel pairs (2j, 2j + 1) meet in lanes differing in bit
      // 3 (pair_mask).  The two lanes of a pair split the tokens: for tokens k, k + 1 the
      // even-channel lane computes output (k, j) from its gate and the partner's up, the odd-channel
      // lane output (k + 1, j) from the partner's gate and its own up -- one shuffle carries both,
      // and every lane evaluates the activation once per two tokens
      const int pair_mask = 8;
      const int NO = act ? N / 2 : N;  // output row length
      grid_dependency_wait();  // y may still be read by the preceding kernel
      int it = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
        const int nt = tile % ntn, mt = tile / ntn;
        const int b = it % L::kAccBufs;
        if (!mbar_wait_warp(&accfull[b], (it / L::kAccBufs) & 1)) {
          report_error(err, kErrTimeoutMma);
          break;
        }
        tc_fence_after_sync();
        if (it == 0 && threadIdx.x == kEpiWarp0 * 32) WQL_STAMP(6);
        const int n = nt * kBM + col_in_tile;
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + b * BN;
#pragma unroll 1
        for (int cc = 0; cc < BN; cc += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + cc, r);
          tmem_ld_wait();
          const int mbase = mt * BN + cc;
          if (act) {
            const bool even = (n & 1) == 0;
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              const float v0 = __uint_as_float(r[k]), v1 = __uint_as_float(r[k + 1]);
              const float got = __shfl_xor_sync(0xffffffffu, even ? v1 : v0, pair_mask);
              const int m = mbase + k + (even ? 0 : 1);
              const __half o = silu_mul_h(even ? v0 : got, even ? got : v1);  // (gate, up)
              if (n < N && m < M) y[(size_t)m * NO + n / 2] = o;
            }
          } else if (n < N) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              if (mbase + k < M) y[(size_t)(mbase + k) * N + n] = __float2half_rn(__uint_as_float(r[k]));
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[b]);
      }
    }
  }

  if (S > 1) {
    // ---------------- split-K: every warp adds the partials of this CTA's columns ----------------
    // the warps that did not drain take their part in (1) here
    if (warp < kDqWarp0 || warp >= kEpiWarp0 + kEpiWarps) {
      if constexpr (L::kOwnRecv)
        cluster_wait();  // (0)
      else
        cluster_phase();  // (1)
    }
    __syncthreads();  // the epilogue warps have seen the receive buffer complete
    // (2) no CTA leaves (freeing the shared memory that its bulk copies read, or that receives
    // another CTA's copies) before every CTA of the cluster has received all of its chunks.  This
    // CTA's chunks have all landed, so it arrives now and waits only before it exits: the adds
    // below overlap the slower peers' receives.
    __syncwarp();
    cluster_arrive_relaxed();
    grid_dependency_wait();  // y may still be read by the preceding kernel
    const int tile = blockIdx.x;
    const int nt = tile % ntn, mt = tile / ntn;
    const int CW = BN / S, rstride = CW + 4;
    const uint32_t recv = L::kOwnRecv ? smem_u32(smem + L::kOffRecv) : smem_u32(smem);
    const int NO = act ? N / 2 : N;
    // Item j: TMEM lane i = j % kBM (a channel), tokens [4 c, 4 c + 4) of this CTA's columns with
    // c = j / kBM.  The 32 lanes of a warp take 32 consecutive TMEM lanes (kThreads and kBM are
    // multiples of 32), so the gate/up pairs meet in the warp as in the epilogue warps, and the
    // stores of one instruction cover 32 channels of one token.  Spreading the additions and stores
    // over all warps instead of the four epilogue warps (a 128 x 128 owner slice: 6.7 -> ? us).
    const int items = kBM * (CW / 4);
    for (int j = threadIdx.x; j < items; j += kThreads) {
      const int i = j % kBM, cl = 4 * (j / kBM);
      const int col_in_tile = tmem_lane_channel(i);
      const int pair_mask = 8;
      const int n = nt * kBM + col_in_tile;
      float4 acc = lds_f4(recv + (uint32_t)((i * rstride + cl) * 4));
      for (int src = 1; src < S; ++src) {  // split order
        const float4 p = lds_f4(recv + (uint32_t)(((src * kBM + i) * rstride + cl) * 4));
        acc.x = __fadd_rn(acc.x, p.x);
        acc.y = __fadd_rn(acc.y, p.y);
        acc.z = __fadd_rn(acc.z, p.z);
        acc.w = __fadd_rn(acc.w, p.w);
      }
      const int m = mt * BN + split * CW + cl;
      const float v[4] = {acc.x, acc.y, acc.z, acc.w};
      if (act) {
        const bool even = (n & 1) == 0;
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const float got = __shfl_xor_sync(0xffffffffu, even ? v[e + 1] : v[e], pair_mask);
          const int mm = m + e + (even ? 0 : 1);
          const __half o = silu_mul_h(even ? v[e] : got, even ? got : v[e + 1]);  // (gate, up)
          if (n < N && mm < M) y[(size_t)mm * NO + n / 2] = o;
        }
      } else if (n < N) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (m + e < M) y[(size_t)(m + e) * N + n] = __float2half_rn(v[e]);
      }
    }
    __syncwarp();
    cluster_wait();  // (2)
  }
  if (threadIdx.x == kEpiWarp0 * 32) WQL_STAMP(10);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, L::kTmemCols);
  if (threadIdx.x == 0) WQL_STAMP(11);
}

template <int BN, int LG, int NACC>
cudaError_t launch_p(const CUtensorMap& tx, const CUtensorMap& tq, const CUtensorMap& ts, const CUtensorMap& tz,
                     int M, int N, int K, __half* y, int act, unsigned* dev_err, cudaStream_t stream) {
  using L = PLayout<BN, LG, NACC>;
  auto kern = w4a16_prefill_kernel<BN, LG, NACC>;
  static std::atomic<bool> attr_set[64];  // per device; racing first calls set the same attribute
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const int ntiles = ((N + kBM - 1) / kBM) * ((M + BN - 1) / BN);
  const int nkb = (K + kBK - 1) / kBK;
  const int sms = num_sms();
  int S = 1;
  // Few tiles: split K over a cluster so that (nearly) every SM streams weights.  Each split keeps
  // at least 512 k; S is a power of two dividing BN into owner column ranges of >= 4 whose exchange
  // buffers fit the stage ring.
  if (2 * ntiles <= sms)
    S = pick_k_split(reinterpret_cast<const void*>(kern), kThreads, L::kBytes, ntiles, nkb * kBK / 512,
                     /*pow2=*/true);
  while (S > 1 && !L::split_fits(S)) S >>= 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = S == 1 ? dim3(ntiles < sms ? ntiles : sms, 1, 1) : dim3(ntiles, S, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = S;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = S == 1 ? 1 : 2;
  return cudaLaunchKernelEx(&cfg, kern, tx, tq, ts, tz, M, N, K, y, act, dev_err);
}

template <int BN, int NACC>
cudaError_t launch_pg(int group, const CUtensorMap& tx, const CUtensorMap& tq, const CUtensorMap& ts,
                      const CUtensorMap& tz, int M, int N, int K, __half* y, int act, unsigned* dev_err,
                      cudaStream_t s) {
  switch (group) {
    case 32:
      return launch_p<BN, 5, NACC>(tx, tq, ts, tz, M, N, K, y, act, dev_err, s);
    case 64:
      return launch_p<BN, 6, NACC>(tx, tq, ts, tz, M, N, K, y, act, dev_err, s);
    default:
      return launch_p<BN, 7, NACC>(tx, tq, ts, tz, M, N, K, y, act, dev_err, s);
  }
}

// One accumulator when every CTA owns at most one tile (the split-K launches always do).
template <int BN>
cudaError_t launch_pa(int group, const CUtensorMap& tx, const CUtensorMap& tq, const CUtensorMap& ts,
                      const CUtensorMap& tz, int M, int N, int K, __half* y, int act, unsigned* dev_err,
                      cudaStream_t s) {
  const int ntiles = ((N + kBM - 1) / kBM) * ((M + BN - 1) / BN);
  if (BN > 128 || ntiles <= num_sms()) return launch_pg<BN, 1>(group, tx, tq, ts, tz, M, N, K, y, act, dev_err, s);
  if constexpr (BN <= 128) return launch_pg<BN, 2>(group, tx, tq, ts, tz, M, N, K, y, act, dev_err, s);
  return cudaErrorInvalidValue;  // not reached
}

}  // namespace

#ifdef WQL_PHASE_TRACE
cudaError_t trace_set_w4a16_prefill(const TraceDesc& d) { return trace_set_local(d); }
#endif

cudaError_t launch_w4a16_prefill(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                                 const uint32_t* qzeros, int M, int K, int N, int group, uint16_t* y, int act,
                                 unsigned* dev_err, cudaStream_t stream, std::string* err) {
  // Token tile: the smallest of 32 / 64 / 128 that holds M; beyond that 256, except up to M = 512
  // where 128-token tiles still fit one wave on the SMs, or where M would leave a 256-tile mostly
  // empty (measured: N = 4096, M = 512: 29 -> 22 us; N = 12288, M = 384: 56 -> 42 us).
  const int ntn = (N + kBM - 1) / kBM;
  int BN = M <= 32 ? 32 : (M <= 64 ? 64 : (M <= 128 ? 128 : 256));
  if (BN == 256 && M <= 512 && (ntn * ((M + 127) / 128) <= num_sms() || (M % 256 != 0 && M % 256 <= 128))) BN = 128;
  // From 257 to 576 tokens, 192-token tiles where they need fewer rounds of CTAs: a round of tiles
  // costs about 0.62 us per 128-k stage at 192 tokens, against 0.70 at 256 and 0.49 at 128 (0.45
  // when CTAs walk several 128-token tiles and overlap their epilogues).  Only tile counts that fill
  // at least half the SMs are compared (fewer go to split-K).  Measured on GB300, K = 4096, us, the
  // previous choice vs 192: M = 512, N = 11008: 51.4 / 45.6; M = 448, N = 12288: 51.2 / 45.7;
  // M = 576, N = 4096: 25.3 / 22.6; M = 576, N = 22016: 102.2 / 91.2; and the cases it leaves
  // alone, e.g. M = 512, N = 4096: 17.9 / 22.6; M = 512, N = 22016: 79.1 / 90.5.
  if (M > 256 && M <= 576) {
    const int sms = num_sms();
    auto tiles = [&](int bn) { return ntn * ((M + bn - 1) / bn); };
    auto cost = [&](int bn) {
      const int rounds = (tiles(bn) + sms - 1) / sms;
      const float per = bn == 128 ? (rounds > 1 ? 0.45f : 0.49f) : (bn == 192 ? 0.62f : 0.70f);
      return rounds * per;
    };
    if (2 * tiles(192) >= sms && cost(192) < cost(BN)) BN = 192;
  }
  const int GR = group >= kBK ? 1 : kBK / group;
  CUtensorMap tx, tq, ts, tz;
  if (!make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, K, M, (uint64_t)K * 2, 64, BN,
                    CU_TENSOR_MAP_SWIZZLE_128B, err) ||
      // rows k = 4a + b as a 3D box {words, a, b}, so that b varies slowest
      !make_tmap_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, qweight, N / 8, K / 4, 4, (uint64_t)N * 2, (uint64_t)N / 2,
                    kStripWords, kBK / 4, 4, CU_TENSOR_MAP_SWIZZLE_64B, err) ||
      !make_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, scales, N, K / group, (uint64_t)N * 2, kBM, GR,
                    CU_TENSOR_MAP_SWIZZLE_NONE, err) ||
      !make_tmap_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, qzeros, N / 8, K / group, (uint64_t)N / 2, kStripWords, GR,
                    CU_TENSOR_MAP_SWIZZLE_NONE, err)) {
    return cudaErrorInvalidValue;
  }
  __half* yh = reinterpret_cast<__half*>(y);
  if (BN == 32) return launch_pa<32>(group, tx, tq, ts, tz, M, N, K, yh, act, dev_err, stream);
  if (BN == 64) return launch_pa<64>(group, tx, tq, ts, tz, M, N, K, yh, act, dev_err, stream);
  if (BN == 192) return launch_pa<192>(group, tx, tq, ts, tz, M, N, K, yh, act, dev_err, stream);
  if (BN == 128) return launch_pa<128>(group, tx, tq, ts, tz, M, N, K, yh, act, dev_err, stream);
  return launch_pa<256>(group, tx, tq, ts, tz, M, N, K, yh, act, dev_err, stream);
}

}  // namespace wql
