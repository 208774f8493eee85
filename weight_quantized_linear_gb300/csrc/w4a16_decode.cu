// w4a16_decode.cu -- AWQ W4A16 GEMM for decode-shaped calls (few tokens, weight-streaming bound).
//
// Computes y[m, n] = sum_k x[m, k] * (q[k, n] - z[k/G, n]) * s[k/G, n] ("LMDeploy ... INT4
// quantisation" tutorial, section 2: per-group asymmetric int4; section 5.1: the engine's fp16 x
// int4 GEMM).  Design for GB300:
//   * The packed weight is streamed exactly once from HBM by TMA (one producer thread), in stages
//     of 64 k-rows x 128 output columns, together with the matching activation, scale and zero
//     tiles.  L2 eviction hint "evict first" keeps the stream from displacing activations.
//   * Eight consumer warps dequantise int4 -> fp16 in registers (PRMT to pair rows k and k+1,
//     LOP3 to splice nibbles into the fp16 pattern 1024 + q, one f16x2 add or fma to subtract
//     1024 + z exactly) and feed the legacy mma.sync.m16n8k16 tensor-core path with the weights
//     as the 16-row operand and the tokens as the 8-column operand ("swap AB").
//   * The per-group scale is applied once per group to fp32 partial sums, not per weight.
//   * Split-K across the CTAs of a thread-block cluster; partial tiles are reduced through
//     distributed shared memory in a fixed order, so results are deterministic and no global
//     scratch is needed.
#include "common.cuh"
#include "internal.h"

namespace wql {
namespace {

constexpr int kBK = 64;            // k rows per stage
constexpr int kStripWords = 16;    // packed words per row of a CTA strip
constexpr int kStripCols = 128;    // output columns per CTA
constexpr int kConsumerWarps = 8;  // 2 column groups (64 columns) x 4 k16 steps
constexpr int kThreads = (kConsumerWarps + 1) * 32;

template <int MT>
struct Layout {
  static constexpr int kXBytes = 8 * MT * kBK * 2;          // token rows x 64 k fp16, 128 B rows
  static constexpr int kWBytes = kBK * kStripWords * 4;     // 64 rows x 64 B
  static constexpr int kSBytes = 2 * kStripCols * 2;        // <= 2 group rows of 128 fp16
  static constexpr int kZBytes = 2 * kStripWords * 4;       // <= 2 group rows of 16 words
  static constexpr int kStage = (kXBytes + kWBytes + kSBytes + kZBytes + 1023) / 1024 * 1024;
  static constexpr int kStages = MT >= 4 ? 6 : 8;
  static constexpr int kPipe = kStages * kStage;
  static constexpr int kRed = 4 * 8 * MT * kStripCols * 4;  // [4 k-steps][tokens][128] fp32
  static constexpr int kData = kPipe > kRed ? kPipe : kRed;
  static constexpr int kBytes = kData + 1024 + 2 * kStages * 8;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Byte offset of packed word j (0..15) of row r in a TMA tile with 64-byte rows and the 64B swizzle
// (16-byte chunk index XOR bits 1..2 of the row).
__device__ __forceinline__ uint32_t wtile_off(int r, int j) {
  return r * 64 + ((((j >> 2) ^ (r >> 1)) & 3) << 4) + (j & 3) * 4;
}

// Zero-point constants for the 8 columns of one packed zero word: even columns are extracted as
// 1024 + q and need -(1024 + z); odd columns as 1024 + 16 q, scaled by 1/16, and need -(64 + z).
__device__ __forceinline__ void zero_consts(uint32_t zw, uint32_t zc[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t z = (zw >> (4 * c)) & 15u;
    zc[c] = (c & 1) ? (0xD400D400u | (z << 4) | (z << 20)) : (0xE400E400u | z | (z << 16));
  }
}

// Four f16x2 registers (q - z) for the 4 columns held in the nibbles of T, exact.
__device__ __forceinline__ void dequant4(uint32_t T, const uint32_t* zc, uint32_t out[4]) {
  const uint32_t kMagic = 0x64006400u, kSixteenth = 0x2C002C00u;
  const uint32_t T8 = T >> 8;
  out[0] = hadd2_u32(and_or(T, 0x000F000Fu, kMagic), zc[0]);
  out[1] = hfma2_u32(and_or(T, 0x00F000F0u, kMagic), kSixteenth, zc[1]);
  out[2] = hadd2_u32(and_or(T8, 0x000F000Fu, kMagic), zc[2]);
  out[3] = hfma2_u32(and_or(T8, 0x00F000F0u, kMagic), kSixteenth, zc[3]);
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_decode_kernel(const __grid_constant__ CUtensorMap tm_x,   // x [M][K] fp16, box {64, 8MT}, SW128
                        const __grid_constant__ CUtensorMap tm_qw,  // qweight [K][N/8], box {16, 64}, SW64
                        const __grid_constant__ CUtensorMap tm_s,   // scales [K/G][N], box {128, GR}
                        const __grid_constant__ CUtensorMap tm_z,   // qzeros [K/G][N/8], box {16, GR}
                        int M, int N, int G, int kblocks, __half* __restrict__ y, unsigned* err) {
  using L = Layout<MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kData);
  uint64_t* empty = full + L::kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int strip = blockIdx.x;
  const int split = blockIdx.y, nsplit = gridDim.y;
  const int m0 = blockIdx.z * 8 * MT;
  const int kb0 = (int)((long long)kblocks * split / nsplit);
  const int kb1 = (int)((long long)kblocks * (split + 1) / nsplit);
  const int GR = G >= kBK ? 1 : kBK / G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbarrier_init();
  }
  __syncthreads();

  float tot[4][MT][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) tot[j][mt][i] = 0.f;

  const int cg = warp & 1, kq = warp >> 1;
  const int g = lane >> 2, t = lane & 3;
  const int wc = cg * 8 + g;  // packed word column within the strip

  if (warp == kConsumerWarps) {
    // ---------------- producer: one thread issues every TMA copy ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_qw);
      tma_prefetch_desc(&tm_s);
      tma_prefetch_desc(&tm_z);
      const uint64_t pol = policy_evict_first();
      const uint32_t bytes = L::kXBytes + L::kWBytes + GR * (kStripCols * 2 + kStripWords * 4);
      int issued = 0;
      bool ok = true;
      grid_dependency_wait();  // activations may come from the preceding kernel
      for (int kb = kb0; kb < kb1; ++kb, ++issued) {
        const int s = issued % L::kStages;
        const uint32_t ph = (issued / L::kStages) & 1;
        if (issued >= L::kStages && !mbar_wait_bounded(&empty[s], ph ^ 1)) {
          report_error(err, kErrTimeoutEmpty);
          ok = false;
          break;
        }
        uint8_t* st = smem + s * L::kStage;
        mbar_arrive_expect_tx(&full[s], bytes);
        const int grow = kb * kBK / G;
        tma_load_2d(st, &tm_x, &full[s], kb * kBK, m0);
        tma_load_2d_hint(st + L::kXBytes, &tm_qw, &full[s], strip * kStripWords, kb * kBK, pol);
        tma_load_2d(st + L::kXBytes + L::kWBytes, &tm_s, &full[s], strip * kStripCols, grow);
        tma_load_2d(st + L::kXBytes + L::kWBytes + L::kSBytes, &tm_z, &full[s], strip * kStripWords, grow);
      }
      // Drain: every issued copy must have landed before shared memory is reused or released.
      const int n = issued < L::kStages ? issued : L::kStages;
      for (int i = issued - n; i < issued; ++i) {
        if (!mbar_wait_bounded(&full[i % L::kStages], (i / L::kStages) & 1)) {
          report_error(err, kErrTimeoutDrain);
          break;
        }
      }
      (void)ok;
    }
  } else {
    // ---------------- consumers: dequantise + tensor-core dot products ----------------
    float acc[4][MT][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[j][mt][i] = 0.f;
    uint32_t zc[8];
    float sc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      zc[c] = 0u;
      sc[c] = 0.f;
    }
    int cur_group = -1;
    const uint32_t sel_lo = (t & 1) ? 0x1054u : 0x5410u;
    const uint32_t sel_hi = (t & 1) ? 0x3276u : 0x7632u;
    const int ra = 16 * kq + 2 * t + (t & 1);      // rows of this thread's k pairs, ordered so that
    const int rb = 16 * kq + 2 * t + 1 - (t & 1);  // the four t lanes hit distinct banks
    const uint32_t offa = wtile_off(ra, wc), offb = wtile_off(rb, wc);
    const uint32_t offc = wtile_off(ra + 8, wc), offd = wtile_off(rb + 8, wc);
    // ldmatrix row addresses for the activation tile (128-byte rows, 128B swizzle)
    uint32_t xoff[(MT + 1) / 2];
#pragma unroll
    for (int p = 0; p < (MT + 1) / 2; ++p) {
      const int mat = lane >> 3;
      const int row = 8 * (2 * p + (mat >> 1)) + (lane & 7);
      const int chunk = 2 * kq + (mat & 1);
      xoff[p] = row * 128 + ((chunk ^ (row & 7)) << 4);
    }

    auto flush = [&]() {
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          tot[j][mt][0] += sc[j] * acc[j][mt][0];
          tot[j][mt][1] += sc[j] * acc[j][mt][1];
          tot[j][mt][2] += sc[j + 4] * acc[j][mt][2];
          tot[j][mt][3] += sc[j + 4] * acc[j][mt][3];
          acc[j][mt][0] = acc[j][mt][1] = acc[j][mt][2] = acc[j][mt][3] = 0.f;
        }
    };

    int it = 0;
    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const int s = it % L::kStages;
      if (!mbar_wait_bounded(&full[s], (it / L::kStages) & 1)) {
        report_error(err, kErrTimeoutFull);
        break;
      }
      const uint32_t st = smem_u32(smem + s * L::kStage);
      const uint32_t wt = st + L::kXBytes;
      const int k0 = kb * kBK + 16 * kq;
      const int grp = k0 / G;
      if (grp != cur_group) {
        if (cur_group >= 0) flush();
        cur_group = grp;
        const int grow = grp - (kb * kBK) / G;
        const uint32_t sbase = wt + L::kWBytes + grow * (kStripCols * 2);
        const uint32_t zbase = wt + L::kWBytes + L::kSBytes + grow * (kStripWords * 4);
        zero_consts(lds_u32(zbase + wc * 4), zc);
        const uint4 sv = lds_u128(sbase + wc * 16);
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&sw[c]));
          sc[2 * c] = f.x;
          sc[2 * c + 1] = f.y;
        }
      }
      // activation fragments (B operand), one pair of registers per token tile
      uint32_t bx[MT][2];
#pragma unroll
      for (int p = 0; p < (MT + 1) / 2; ++p) {
        if (2 * p + 1 < MT) {
          ldmatrix_x4(st + xoff[p], bx[2 * p][0], bx[2 * p][1], bx[2 * p + 1][0], bx[2 * p + 1][1]);
        } else {
          ldmatrix_x2(st + xoff[p], bx[2 * p][0], bx[2 * p][1]);
        }
      }
      // weight fragments (A operand): rows 2t, 2t+1 and 2t+8, 2t+9 of this k16 step
      const uint32_t w0 = lds_u32(wt + offa), w1 = lds_u32(wt + offb);
      const uint32_t w2 = lds_u32(wt + offc), w3 = lds_u32(wt + offd);
      uint32_t lo[4], hi[4], lo2[4], hi2[4];
      dequant4(prmt(w0, w1, sel_lo), zc, lo);
      dequant4(prmt(w0, w1, sel_hi), zc + 4, hi);
      dequant4(prmt(w2, w3, sel_lo), zc, lo2);
      dequant4(prmt(w2, w3, sel_hi), zc + 4, hi2);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t a[4] = {lo[j], hi[j], lo2[j], hi2[j]};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma_f16_16816(acc[j][mt], a, bx[mt][0], bx[mt][1]);
      }
    }
    if (cur_group >= 0) flush();
  }

  // ---------------- reduction over the 4 k-step warps and the cluster's k splits ----------------
  __syncthreads();  // all stages consumed and drained: the pipeline memory is free
  float* red = reinterpret_cast<float*>(smem);
  constexpr int kE = 8 * MT * kStripCols;  // elements of one partial tile
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = 8 * mt + 2 * t + (i & 1);
          const int col = 8 * wc + j + 4 * (i >> 1);
          red[kq * kE + row * kStripCols + col] = tot[j][mt][i];
        }
  }
  cluster_sync();
  {
    const uint32_t rank = cluster_ctarank();
    const int nq = kE / 4;
    const int f0 = (int)((long long)nq * rank / nsplit), f1 = (int)((long long)nq * (rank + 1) / nsplit);
    for (int f = f0 + threadIdx.x; f < f1; f += kThreads) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < nsplit; ++q) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float4 p = ld_cluster_f4(map_cluster(red + w * kE + 4 * f, q));
          v.x += p.x;
          v.y += p.y;
          v.z += p.z;
          v.w += p.w;
        }
      }
      const int row = (4 * f) / kStripCols, col = (4 * f) % kStripCols;
      const int m = m0 + row, n = strip * kStripCols + col;
      if (m < M && n < N) {
        __half2 h01 = __floats2half2_rn(v.x, v.y), h23 = __floats2half2_rn(v.z, v.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&h01);
        pk.y = *reinterpret_cast<uint32_t*>(&h23);
        *reinterpret_cast<uint2*>(y + (size_t)m * N + n) = pk;
      }
    }
  }
  cluster_sync();  // keep this CTA's partial tile alive until every peer has read it
}

template <int MT>
cudaError_t launch_mt(const CUtensorMap& tx, const CUtensorMap& tq, const CUtensorMap& ts,
                      const CUtensorMap& tz, int M, int N, int G, int kblocks, __half* y, unsigned* dev_err,
                      cudaStream_t stream) {
  using L = Layout<MT>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(w4a16_decode_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int strips = (N + kStripCols - 1) / kStripCols;
  const int mblocks = (M + 8 * MT - 1) / (8 * MT);
  const int target = 2 * num_sms();
  int S = (target + strips * mblocks - 1) / (strips * mblocks);
  if (S > 8) S = 8;
  if (S > kblocks) S = kblocks;
  if (S < 1) S = 1;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(strips, S, mblocks);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = 1;
  attrs[na].val.clusterDim.y = S;
  attrs[na].val.clusterDim.z = 1;
  ++na;
  attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, w4a16_decode_kernel<MT>, tx, tq, ts, tz, M, N, G, kblocks, y, dev_err);
}

}  // namespace

cudaError_t launch_w4a16_decode(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                                const uint32_t* qzeros, int M, int K, int N, int group, uint16_t* y,
                                unsigned* dev_err, cudaStream_t stream, std::string* err) {
  const int MT = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
  const int GR = group >= kBK ? 1 : kBK / group;
  CUtensorMap tx, tq, ts, tz;
  if (!make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, K, M, (uint64_t)K * 2, kBK, 8 * MT,
                    CU_TENSOR_MAP_SWIZZLE_128B, err) ||
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
  switch (MT) {
    case 1:
      return launch_mt<1>(tx, tq, ts, tz, M, N, group, kblocks, yh, dev_err, stream);
    case 2:
      return launch_mt<2>(tx, tq, ts, tz, M, N, group, kblocks, yh, dev_err, stream);
    default:
      return launch_mt<4>(tx, tq, ts, tz, M, N, group, kblocks, yh, dev_err, stream);
  }
}

}  // namespace wql
