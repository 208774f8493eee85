// w4a16_decode.cu -- AWQ W4A16 GEMM for decode-shaped calls (few tokens, weight-streaming bound).
//
// Computes y[m, n] = sum_k x[m, k] * (q[k, n] - z[k/G, n]) * s[k/G, n] ("LMDeploy ... INT4
// quantisation" tutorial, section 2: per-group asymmetric int4; section 5.1: the engine's fp16 x
// int4 GEMM).  Design for GB300:
//   * The packed weight is streamed exactly once from HBM by TMA (one producer thread), in stages
//     of 128 k-rows x 128 output columns with the matching scale and zero-point rows and the
//     stage's activation slab (one 3D copy).  "Evict first" L2 hints on the weight stream.
//   * Programmatic dependent launch: each CTA issues its weight copies before waiting for the
//     previous kernel; only the activation copies wait.  It lets the next kernel launch as soon as
//     those activation copies are issued, so the next layer's CTAs stream their weights during
//     this layer's arithmetic and reduction without delaying its activations.
//   * Consumer warps: two column groups of 64 outputs x four stage lanes for 8-token blocks, two
//     lanes for 16-token blocks (lane l owns every stage i with i % lanes == l, so every group is
//     reduced by a single warp).  They feed the legacy
//     mma.sync.m16n8k16 tensor-core path with the weights as the 16-row operand and the tokens as
//     the 8-column operand ("swap AB").  The int4 codes enter the MMA as the exact fp16 values
//     1024 + q (or 1024 + 16 q): a transposed ldmatrix pairs rows k and k+1 of the packed tile in
//     one register, one LOP3 per two weights splices the nibbles into the fp16 bit pattern.  Offset, zero point and scale are applied once per
//     group to the fp32 partial sums:
//         sum_k (q - z) x = D - (1024 + z) sum_k x       (D = sum_k (1024 + q) x)
//         sum_k (q - z) x = D / 16 - (64 + z) sum_k x    (D = sum_k (1024 + 16 q) x)
//     with sum_k x of each token taken from one extra MMA against an all-ones operand.
//   * Split-K across the CTAs of a thread-block cluster: every consumer thread sends its partial
//     sums straight into the owning CTA's receive buffer with st.async, which completes
//     transaction bytes on the owner's mbarrier; owners add the partials in a fixed order.
//     Deterministic and free of global scratch.  Cluster barrier phase 0 (arrive at start, wait
//     before the first remote store) guarantees every peer is initialised; phase 1 (arrive once
//     the own slice is complete, wait before exit) keeps every CTA alive until all stores landed.
#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "trace.cuh"

namespace wql {
namespace {

constexpr int kBK = 128;           // k rows per stage (a multiple of every group size)
constexpr int kStripWords = 16;    // packed words per row of a CTA strip
constexpr int kStripCols = 128;    // output columns per CTA

// Stage lanes: four for blocks of 8 tokens, two for blocks of 16.  With two lanes a 16-token CTA
// has 160 threads, so it and a CTA of the next layer fit one SM's register file together (the
// next layer's CTAs stream their weights while this one computes).
template <int MT>
struct Warps {
  static constexpr int kLanes = MT <= 1 ? 4 : 2;
  static constexpr int kConsumerWarps = 2 * kLanes;  // two column groups per lane
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
};

template <int MT, int LG>
struct Layout {
  static constexpr int G = 1 << LG;
  static constexpr int kGR = G >= kBK ? 1 : kBK / G;      // groups per stage
  static constexpr int kLanes = Warps<MT>::kLanes;
  // Slot s of the ring is always served by stage lane s % kLanes, so a lane can never lap another
  // lane on a slot (the parity-based barrier waits rely on it): the depth is a multiple of kLanes.
  static constexpr int kStages = 8;
  static_assert(kStages % kLanes == 0, "ring depth must be a multiple of the lane count");
  static constexpr int kSlab = 8 * MT * 128;              // token rows x 64 k fp16 (128-byte rows)
  static constexpr int kXBytes = 2 * kSlab;               // two 64-k slabs per stage
  static constexpr int kWBytes = kBK * kStripWords * 4;   // 128 rows x 64 B
  static constexpr int kSBytes = kGR * kStripCols * 2;
  static constexpr int kZBytes = kGR * kStripWords * 4;
  // A stage is [activation slabs | packed tile], 1024-byte aligned for the 128B swizzle; its
  // scale and zero-point rows sit in a separate array, so the stages carry no padding.
  static constexpr int kStage = kXBytes + kWBytes;
  static_assert(kStage % 1024 == 0, "stages must keep the 128B-swizzled slabs 1024-byte aligned");
  static constexpr int kSZ = (kSBytes + kZBytes + 127) / 128 * 128;
  static constexpr int kE = 8 * MT * kStripCols;          // elements of one partial tile
  static constexpr int kNQ = kE / 4;                      // float4s of one partial tile
  static constexpr uint32_t kTx = kXBytes + kWBytes + kSBytes + kZBytes;
  // shared memory map: [stages (1024-aligned)] [scale/zero rows per stage] [receive buffer] [barriers]
  static constexpr int kOffSZ = kStages * kStage;
  static constexpr int kOffRecv = kOffSZ + kStages * kSZ;
  static int bytes(int S) {
    const int lmax = (kNQ + S - 1) / S;
    return kOffRecv + S * lmax * 16 + (2 * kStages + 1) * 8 + 1024;
  }
};

// Shared-memory footprint of every decode launch with group size 2^LG: the largest over both token
// blocks and every split, as long as two such CTAs still fit one SM (0 otherwise: each launch then
// takes its own size).  Back-to-back layers keep one CTA of each of two consecutive layers per SM
// only when the block scheduler sees alike CTAs; with footprints that differ between 8- and
// 16-token layers, a change of token count left some SMs with two CTAs of one layer for the rest
// of the sequence (measured: 48 q_proj layers at M = 1 then 48 at M = 16, 479 -> 402 us).
template <int LG>
int common_footprint() {
  static std::atomic<int> cached{-1};  // racing first calls store the same value
  int bytes = cached.load(std::memory_order_relaxed);
  if (bytes < 0) {
    int f = 0;
    for (int S = 1; S <= 8; ++S) {
      f = Layout<1, LG>::bytes(S) > f ? Layout<1, LG>::bytes(S) : f;
      f = Layout<2, LG>::bytes(S) > f ? Layout<2, LG>::bytes(S) : f;
    }
    int dev = 0, per_sm = 0, reserved = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    bytes = 2 * (f + reserved) <= per_sm ? f : 0;
    cached.store(bytes, std::memory_order_relaxed);
  }
  return bytes;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// The four f16x2 MMA operands held in the nibbles of T: columns 0 and 2 as 1024 + q, columns 1 and
// 3 as 1024 + 16 q (both exact).
__device__ __forceinline__ void splice4(uint32_t T, uint32_t out[4]) {
  const uint32_t kMagic = 0x64006400u;
  const uint32_t T8 = T >> 8;
  out[0] = and_or(T, 0x000F000Fu, kMagic);
  out[1] = and_or(T, 0x00F000F0u, kMagic);
  out[2] = and_or(T8, 0x000F000Fu, kMagic);
  out[3] = and_or(T8, 0x00F000F0u, kMagic);
}

template <int MT, int LG>
__global__ void __launch_bounds__(Warps<MT>::kThreads, 2)
    w4a16_decode_kernel(const __grid_constant__ CUtensorMap tm_x,   // x: 3D {64, M, K/64} box {64, 8MT, 2}, or
                                                                    //    2D {K, M} box {64, 8MT} (x3d == 0)
                        const __grid_constant__ CUtensorMap tm_qw,  // qweight [K][N/8], box {16, 128}, SW64
                        const __grid_constant__ CUtensorMap tm_s,   // scales [K/G][N], box {128, GR}
                        const __grid_constant__ CUtensorMap tm_z,   // qzeros [K/G][N/8], box {16, GR}
                        int M, int N, int kblocks, int x3d, __half* __restrict__ y, int act, unsigned* err) {
  using L = Layout<MT, LG>;
  // phase stamps (trace builds only): 0 start, 1 dependency resolved, 2 first stage landed, 3 last
  // consumer warp done, 4 lanes folded, 5 own slice received, 6 end
  WQL_TRACE_ROW(y);
  if (threadIdx.x == 0) {
    WQL_STAMP(0);
    WQL_STAMP_SMID();
  }
  constexpr int kLanes = L::kLanes;
  constexpr int kConsumerWarps = Warps<MT>::kConsumerWarps;
  constexpr int kThreads = Warps<MT>::kThreads;
  constexpr int G = L::G;
  constexpr int kGR = L::kGR;
  constexpr int kStages = L::kStages;
  constexpr int kStepsPerGroup = (G >= kBK ? kBK : G) / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int strip = blockIdx.x;
  const int nsplit = gridDim.y;
  const int m0 = blockIdx.z * 8 * MT;
  const int kb0 = (int)((long long)kblocks * blockIdx.y / nsplit);
  const int kb1 = (int)((long long)kblocks * (blockIdx.y + 1) / nsplit);
  const int nkb = kb1 - kb0;
  const int lmax = (L::kNQ + nsplit - 1) / nsplit;  // owner r holds float4s [r lmax, min((r+1) lmax, nq))
  const uint32_t rank = cluster_ctarank();

  float4* recv = reinterpret_cast<float4*>(smem + L::kOffRecv);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffRecv + nsplit * lmax * 16);
  uint64_t* empty = full + kStages;
  uint64_t* recv_full = empty + kStages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);  // the two column-group warps of the slot's lane
    }
    mbar_init(recv_full, 1);
    fence_mbarrier_init();
    const int own0 = (int)rank * lmax, own1 = own0 + lmax < L::kNQ ? own0 + lmax : L::kNQ;
    // the owner's slice arrives once from every CTA of the cluster as st.async transaction bytes
    mbar_arrive_expect_tx(recv_full, (uint32_t)(nsplit * (own1 > own0 ? own1 - own0 : 0) * 16));
  }
  __syncwarp();
  cluster_arrive_relaxed();  // phase 0: this CTA's receive buffer and barriers are initialised
  __syncthreads();

  const int cg = warp & 1, kq = warp >> 1;
  const int g = lane >> 2, t = lane & 3;

  if (warp == kConsumerWarps) {
    // ---------------- producer: one thread issues every TMA copy ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_qw);
      tma_prefetch_desc(&tm_s);
      tma_prefetch_desc(&tm_z);
      const uint64_t pol = policy_evict_first();
      auto issue_weights = [&](int i) {
        const int s = i % kStages, kb = kb0 + i;
        uint8_t* st = smem + s * L::kStage + L::kXBytes;
        uint8_t* sz = smem + L::kOffSZ + s * L::kSZ;
        const int grow = (kb * kBK) >> LG;
        mbar_arrive_expect_tx(&full[s], L::kTx);
        tma_load_2d_hint(st, &tm_qw, &full[s], strip * kStripWords, kb * kBK, pol);
        tma_load_2d_hint(sz, &tm_s, &full[s], strip * kStripCols, grow, pol);
        tma_load_2d_hint(sz + L::kSBytes, &tm_z, &full[s], strip * kStripWords, grow, pol);
      };
      auto issue_x = [&](int i) {
        const int s = i % kStages, kb = kb0 + i;
        uint8_t* st = smem + s * L::kStage;
        if (x3d) {
          tma_load_3d(st, &tm_x, &full[s], 0, m0, 2 * kb);
        } else {
          tma_load_2d(st, &tm_x, &full[s], kb * kBK, m0);
          tma_load_2d(st + L::kSlab, &tm_x, &full[s], kb * kBK + 64, m0);
        }
      };
      // prologue: weights first (independent of the previous kernel), then activations
      const int pro = nkb < kStages ? nkb : kStages;
      for (int i = 0; i < pro; ++i) issue_weights(i);
      grid_dependency_wait();  // activations may come from the preceding kernel
      WQL_STAMP(1);
      for (int i = 0; i < pro; ++i) issue_x(i);
      // Only now may the next kernel launch: its CTAs share these SMs and open with a burst of
      // weight copies, which would otherwise queue in the SM's TMA unit ahead of the activation
      // copies above, on this layer's critical path (q_proj M = 1 back to back: 5.07 -> 3.66 us).
      grid_dependents_launch();
      int issued = pro;
      for (; issued < nkb; ++issued) {
        const int s = issued % kStages;
        if (!mbar_wait_bounded(&empty[s], ((issued / kStages) & 1) ^ 1)) {
          report_error(err, kErrTimeoutEmpty);
          break;
        }
        issue_weights(issued);
        issue_x(issued);
      }
      // Drain: every issued copy must have landed before shared memory is reused or released.
      const int n = issued < kStages ? issued : kStages;
      for (int i = issued - n; i < issued; ++i) {
        if (!mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1)) {
          report_error(err, kErrTimeoutDrain);
          break;
        }
      }
    }
    __syncwarp();
    cluster_wait();  // phase 0
  } else {
    // ---------------- consumers: splice codes + tensor-core dot products ----------------
    cluster_wait();  // phase 0, while the first activations are still in flight
    float tot[4][MT][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) tot[j][mt][i] = 0.f;
    const uint32_t kOnes[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};
    // The packed tile's rows are k (64 bytes = 16 words = 128 columns, 64B swizzle: the 16-byte chunk
    // index is XORed with bits 1..2 of the row).  One transposed ldmatrix per k16 step loads four
    // 8 x 8 b16 matrices: lane 4g + t receives half-word g of a 16-byte chunk (four codes, columns
    // 4g .. 4g + 3 of the chunk's 32) for k rows 2t and 2t + 1 -- the row pairing the MMA's A
    // fragment wants.  Matrices: (k 0-7, chunk 2cg), (k 0-7, chunk 2cg + 1), (k 8-15, chunk 2cg),
    // (k 8-15, chunk 2cg + 1).  Row address of this lane for step 0; step u sits 16 rows further.
    const int mi = lane >> 3, wr = 8 * (mi >> 1) + (lane & 7);
    const uint32_t woff = wr * 64 + ((((2 * cg + (mi & 1)) ^ (wr >> 1)) & 3) << 4);
    // MMA row g holds column c0 + j of MMA j, row g + 8 column c0 + 32 + j
    const int c0 = 64 * cg + 4 * g;
    // ldmatrix row addresses for chunk pair u2 (k16 step) within one activation slab (128-byte rows,
    // 128B swizzle); matrices: (tokens 0-7, chunks 2u2, 2u2+1), then the next token tile
    uint32_t xoff[4][(MT + 1) / 2];
#pragma unroll
    for (int u2 = 0; u2 < 4; ++u2)
#pragma unroll
      for (int p = 0; p < (MT + 1) / 2; ++p) {
        const int mat = lane >> 3;
        const int row = 8 * (2 * p + (mat >> 1)) + (lane & 7);
        const int chunk = 2 * u2 + (mat & 1);
        xoff[u2][p] = row * 128 + ((chunk ^ (row & 7)) << 4);
      }

    for (int i = kq; i < nkb; i += kLanes) {
      const int s = i % kStages;
      if (!mbar_wait_bounded(&full[s], (i / kStages) & 1)) {
        report_error(err, kErrTimeoutFull);
        break;
      }
      if (i == 0 && threadIdx.x == 0) WQL_STAMP(2);
      const uint32_t xt = smem_u32(smem + s * L::kStage);
      const uint32_t wt = xt + L::kXBytes;
      const uint32_t sbase = smem_u32(smem + L::kOffSZ + s * L::kSZ), zbase = sbase + L::kSBytes;
#pragma unroll
      for (int gi = 0; gi < kGR; ++gi) {
        float acc[4][MT][4];
        float sx[MT][4];
#pragma unroll
        for (int uu = 0; uu < kStepsPerGroup; ++uu) {
          const int u = gi * kStepsPerGroup + uu;  // k16 step within the stage (0..7)
          const int hb = u >> 2, u2 = u & 3;       // activation slab and chunk pair
          uint32_t bx[MT][2];
#pragma unroll
          for (int p = 0; p < (MT + 1) / 2; ++p) {
            if (2 * p + 1 < MT)
              ldmatrix_x4(xt + hb * L::kSlab + xoff[u2][p], bx[2 * p][0], bx[2 * p][1], bx[2 * p + 1][0],
                          bx[2 * p + 1][1]);
            else
              ldmatrix_x2(xt + hb * L::kSlab + xoff[u2][p], bx[2 * p][0], bx[2 * p][1]);
          }
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(wt + u * 1024 + woff, r0, r1, r2, r3);
          uint32_t lo[4], hi[4], lo2[4], hi2[4];
          splice4(r0, lo);
          splice4(r1, hi);
          splice4(r2, lo2);
          splice4(r3, hi2);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t a[4] = {lo[j], hi[j], lo2[j], hi2[j]};
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              if (uu == 0) acc[j][mt][0] = acc[j][mt][1] = acc[j][mt][2] = acc[j][mt][3] = 0.f;
              mma_f16_16816(acc[j][mt], a, bx[mt][0], bx[mt][1]);
            }
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if (uu == 0) sx[mt][0] = sx[mt][1] = sx[mt][2] = sx[mt][3] = 0.f;
            mma_f16_16816(sx[mt], kOnes, bx[mt][0], bx[mt][1]);
          }
        }
        // group epilogue: tot += ca * acc - cb * sx per column
        // coefficients of column c0 + 32 h + j at [j + 4 h]: its zero point is nibble 4 (g & 1) + j of
        // packed word (c0 + 32 h) / 8, its scale the fp16 at column c0 + 32 h
        float ca[8], cb[8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t zw = lds_u32(zbase + gi * (kStripWords * 4) + ((c0 + 32 * h) >> 3) * 4) >> (16 * (g & 1));
          const uint2 sv = lds_u64(sbase + gi * (kStripCols * 2) + (c0 + 32 * h) * 2);
          const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&sv.x));
          const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&sv.y));
          const float sc4[4] = {f01.x, f01.y, f23.x, f23.y};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // 1024 + z (j even: codes entered as 1024 + q) or 64 + z (j odd: 1024 + 16 q), built
            // directly as fp32 bit patterns
            const uint32_t z = (zw >> (4 * j)) & 15u;
            const uint32_t zb = (j & 1) ? (0x42800000u | (z << 17)) : (0x44800000u | (z << 13));
            ca[j + 4 * h] = (j & 1) ? sc4[j] * 0.0625f : sc4[j];
            cb[j + 4 * h] = sc4[j] * __uint_as_float(zb);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int cc = j + 4 * (e >> 1);
              tot[j][mt][e] = fmaf(ca[cc], acc[j][mt][e], fmaf(-cb[cc], sx[mt][e & 1], tot[j][mt][e]));
            }
      }
      // The stage was read through ordinary shared-memory loads (the generic proxy); TMA refills it
      // through the async proxy once the producer sees this release.  An mbarrier release alone does
      // not order generic-proxy reads before async-proxy writes: without this fence a refill could
      // land while an earlier read was still being performed (seen as 1-4 % of back-to-back calls
      // with wrong partial sums at N = 22016 under cluster split-K).
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (lane == 0) WQL_STAMP_MAX(3);

    // Fold the lanes' partials in shared memory first.  Once all consumer warps pass this
    // named barrier every stage has been consumed and every issued copy has landed (each one was
    // waited for by its lane), so the pipeline memory is free for staging.
    // Float4 f = 32 row + c of a partial tile sits at f ^ (row & 7): without the swizzle the four
    // t lanes of every quarter warp store to the same bank group (4-way conflicts on 16-byte stores,
    // measured as 0.3 us of queued stores ahead of the loads below at 8 tokens).
    named_barrier_sync(1, kConsumerWarps * 32);
    float4* stage4 = reinterpret_cast<float4*>(smem);  // [lane][swizzled float4 index]
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 8 * mt + 2 * t + (e & 1);
        const int col = c0 + 32 * (e >> 1);
        stage4[kq * L::kNQ + (((row * kStripCols + col) >> 2) ^ (row & 7))] =
            make_float4(tot[0][mt][e], tot[1][mt][e], tot[2][mt][e], tot[3][mt][e]);
      }
    named_barrier_sync(1, kConsumerWarps * 32);
    if (threadIdx.x == 0) WQL_STAMP(4);
    // split-K: send each folded float4 to its owner CTA
    const uint32_t recv_base = smem_u32(recv);
    const uint32_t bar_local = smem_u32(recv_full);
    for (int f = threadIdx.x; f < L::kNQ; f += kConsumerWarps * 32) {
      const int fs = f ^ ((f >> 5) & 7);
      float4 v = stage4[fs];
#pragma unroll
      for (int q = 1; q < kLanes; ++q) {  // lane order
        const float4 p = stage4[q * L::kNQ + fs];
        v.x += p.x;
        v.y += p.y;
        v.z += p.z;
        v.w += p.w;
      }
      const int owner = f / lmax;
      const uint32_t slot = recv_base + (uint32_t)(((int)rank * lmax + (f - owner * lmax)) * 16);
      st_async_f4(map_cluster_addr(slot, owner), v, map_cluster_addr(bar_local, owner));
    }
  }

  // ---------------- owners: add the partials of their slice in a fixed order ----------------
  const bool received = mbar_wait_bounded(recv_full, 0);
  if (!received) report_error(err, kErrTimeoutMma);
  if (threadIdx.x == 0) WQL_STAMP(5);
  __syncwarp();
  // phase 1: this CTA's slice is complete (an execution barrier only: the receive barrier has
  // already ordered the data, so no release fence is needed)
  cluster_arrive_relaxed();
  if (received) {
    const int f0 = (int)rank * lmax;
    const int f1 = f0 + lmax < L::kNQ ? f0 + lmax : L::kNQ;
    for (int f = f0 + threadIdx.x; f < f1; f += kThreads) {
      float4 v = recv[f - f0];
      for (int q = 1; q < nsplit; ++q) {
        const float4 p = recv[q * lmax + (f - f0)];
        v.x += p.x;
        v.y += p.y;
        v.z += p.z;
        v.w += p.w;
      }
      const int row = (4 * f) / kStripCols, col = (4 * f) % kStripCols;
      const int m = m0 + row, n = strip * kStripCols + col;
      if (m < M && n < N) {
        if (act) {  // channels n, n + 1 and n + 2, n + 3 are (gate, up) pairs: outputs n / 2, n / 2 + 1
          *reinterpret_cast<__half2*>(y + (size_t)m * (N / 2) + n / 2) =
              __halves2half2(silu_mul_h(v.x, v.y), silu_mul_h(v.z, v.w));
        } else {
          __half2 h01 = __floats2half2_rn(v.x, v.y), h23 = __floats2half2_rn(v.z, v.w);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t*>(&h01);
          pk.y = *reinterpret_cast<uint32_t*>(&h23);
          *reinterpret_cast<uint2*>(y + (size_t)m * N + n) = pk;
        }
      }
    }
  }
  __syncwarp();
  cluster_wait();  // phase 1: no CTA exits before every slice in the cluster is complete
  if (threadIdx.x == 0) WQL_STAMP(6);
}

template <int MT, int LG>
cudaError_t launch_mt(const CUtensorMap& tx, int x3d, const CUtensorMap& tq, const CUtensorMap& ts,
                      const CUtensorMap& tz, int M, int N, int kblocks, __half* y, int act, unsigned* dev_err,
                      cudaStream_t stream) {
  using L = Layout<MT, LG>;
  constexpr int kThreads = Warps<MT>::kThreads;
  auto kern = w4a16_decode_kernel<MT, LG>;
  static std::atomic<bool> attr_set[64];  // per device; racing first calls set the same attribute
  int dev = 0;
  cudaGetDevice(&dev);
  const int common = common_footprint<LG>();
  int max_bytes = common;  // otherwise the largest over the cluster sizes (the receive buffer varies)
  if (!common)
    for (int S = 1; S <= 8; ++S) max_bytes = L::bytes(S) > max_bytes ? L::bytes(S) : max_bytes;
  if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_bytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const int strips = (N + kStripCols - 1) / kStripCols;
  const int mblocks = (M + 8 * MT - 1) / (8 * MT);
  const int S = pick_k_split(reinterpret_cast<const void*>(kern), kThreads, max_bytes, strips * mblocks, kblocks,
                             /*pow2=*/false, /*balanced=*/true);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(strips, S, mblocks);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = common ? common : L::bytes(S);
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
  return cudaLaunchKernelEx(&cfg, kern, tx, tq, ts, tz, M, N, kblocks, x3d, y, act, dev_err);
}

template <int MT>
cudaError_t launch_g(int group, const CUtensorMap& tx, int x3d, const CUtensorMap& tq, const CUtensorMap& ts,
                     const CUtensorMap& tz, int M, int N, int kblocks, __half* y, int act, unsigned* dev_err,
                     cudaStream_t s) {
  switch (group) {
    case 32:
      return launch_mt<MT, 5>(tx, x3d, tq, ts, tz, M, N, kblocks, y, act, dev_err, s);
    case 64:
      return launch_mt<MT, 6>(tx, x3d, tq, ts, tz, M, N, kblocks, y, act, dev_err, s);
    default:
      return launch_mt<MT, 7>(tx, x3d, tq, ts, tz, M, N, kblocks, y, act, dev_err, s);
  }
}

}  // namespace

#ifdef WQL_PHASE_TRACE
cudaError_t trace_set_w4a16_decode(const TraceDesc& d) { return trace_set_local(d); }
#endif

cudaError_t launch_w4a16_decode(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                                const uint32_t* qzeros, int M, int K, int N, int group, uint16_t* y, int act,
                                unsigned* dev_err, cudaStream_t stream, std::string* err) {
  const int MT = M <= 8 ? 1 : 2;  // larger M runs as several 16-token blocks
  const int GR = group >= kBK ? 1 : kBK / group;
  CUtensorMap tx, tq, ts, tz;
  // Activations: 64-k slabs of 8 MT token rows, 128-byte rows with the 128B swizzle.  With K a
  // multiple of 64, one 3D copy fetches both slabs of a stage; otherwise one 2D copy per slab.
  const int x3d = (K % 64 == 0) ? 1 : 0;
  const bool okx = x3d ? make_tmap_3d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, 64, M, K / 64, (uint64_t)K * 2, 128, 64,
                                      8 * MT, 2, CU_TENSOR_MAP_SWIZZLE_128B, err)
                       : make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, K, M, (uint64_t)K * 2, 64, 8 * MT,
                                      CU_TENSOR_MAP_SWIZZLE_128B, err);
  if (!okx ||
      !make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, qweight, N / 8, K, (uint64_t)N / 2, kStripWords, kBK,
                    CU_TENSOR_MAP_SWIZZLE_64B, err) ||
      !make_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, scales, N, K / group, (uint64_t)N * 2, kStripCols, GR,
                    CU_TENSOR_MAP_SWIZZLE_NONE, err) ||
      !make_tmap_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, qzeros, N / 8, K / group, (uint64_t)N / 2, kStripWords,
                    GR, CU_TENSOR_MAP_SWIZZLE_NONE, err)) {
    return cudaErrorInvalidValue;
  }
  const int kblocks = (K + kBK - 1) / kBK;
  __half* yh = reinterpret_cast<__half*>(y);
  if (MT == 1) return launch_g<1>(group, tx, x3d, tq, ts, tz, M, N, kblocks, yh, act, dev_err, stream);
  return launch_g<2>(group, tx, x3d, tq, ts, tz, M, N, kblocks, yh, act, dev_err, stream);
}

}  // namespace wql
