// epilogue.cuh -- optional terms of the int8 / fp8 GEMM's epilogue ("LMDeploy W8A8 quantisation
// guide", inference kernels: the _linear_add variant of matmul_kernel_dynamic_quant fuses a bias and
// a residual into c = c * rms_scale * linear_scale).  The sum is taken in fp32, left to right, after
// the scaled value and before the single rounding to fp16:
//     y[m, n] = fp16(((acc * xs[m]) * ws[n] + bias[n]) + residual[m, n])
// A null pointer leaves its term out (adding 0.0 would turn a -0.0 result into +0.0).
//
// The decode kernels load a thread's four terms with one 8-byte load each.  The tcgen05 kernels stage
// their output through shared memory (BoxStage below), where TMA has brought the residual ahead of
// time.  y may be the residual buffer itself: every output element is computed from its own residual
// value, loaded before the output is written.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace wql {

struct EpilogueAdd {
  const __half* bias;      // [N], or null
  const __half* residual;  // [M, N] row-major, or null; may be the output y itself
};

// u + b + r with the terms already widened to fp32; a term whose pointer is null is not added.
__device__ __forceinline__ float add_terms(float u, const EpilogueAdd& ea, float b, float r) {
  if (ea.bias) u = __fadd_rn(u, b);
  if (ea.residual) u = __fadd_rn(u, r);
  return u;
}

// Four consecutive fp16 values (8-byte aligned) widened to fp32.
__device__ __forceinline__ void load_half4(const __half* p, float (&v)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  const __half2 lo = *reinterpret_cast<const __half2*>(&raw.x), hi = *reinterpret_cast<const __half2*>(&raw.y);
  v[0] = __low2float(lo);
  v[1] = __high2float(lo);
  v[2] = __low2float(hi);
  v[3] = __high2float(hi);
}

// Output staging of one epilogue warp of the tcgen05 GEMMs.  The warp owns 32 output channels (its
// lanes) and writes a tile's tokens in boxes of 32 tokens x 32 channels, fp16, row = token, held in
// one of kBufs shared-memory buffers and stored to y by TMA (the part outside [M, N] is clipped).
// With a fused residual, TMA first loads the box's residual values into the buffer, up to kBufs boxes
// ahead, and the outputs overwrite them in place.  All calls are made by the whole warp.
template <int kBufs>
struct BoxStage {
  __half* box;               // [kBufs][32][32]
  uint64_t* bar;             // [kBufs] residual box landed (initialised with count 1)
  const CUtensorMap* tm_y;   // y fp16 [M][N], box {32, 32}
  const CUtensorMap* tm_r;   // residual fp16 [M][N], box {32, 32}
  bool has_res;
  uint32_t phase;            // parity of the next wait on bar[i], bit i
  uint32_t pend;             // residual loads issued and not yet waited for, bit per buffer
  int seq;                   // boxes begun by this warp; box j of the current tile uses (seq0 + j) % kBufs
  int seq0, issued, nbox, n0, m0;

  __device__ __forceinline__ void init(__half* box_, uint64_t* bar_, const CUtensorMap* ty, const CUtensorMap* tr,
                                       bool res) {
    box = box_, bar = bar_, tm_y = ty, tm_r = tr, has_res = res;
    phase = pend = 0u;
    seq = seq0 = issued = nbox = n0 = m0 = 0;
  }
  __device__ __forceinline__ void issue(int j, int lane) {
    const int buf = (seq0 + j) % kBufs;
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar[buf], 32 * 32 * 2);
      tma_load_2d(box + buf * 32 * 32, tm_r, &bar[buf], n0, m0 + 32 * j);
    }
    pend |= 1u << buf;
  }
  // Start a tile whose boxes cover channels n0_ .. n0_ + 31 and tokens m0_ .. m0_ + 32 nbox_ - 1:
  // the first kBufs residual boxes are requested at once (call it well before the accumulator is
  // ready, so that they land meanwhile).
  __device__ __forceinline__ void begin(int n0_, int m0_, int nbox_, int lane) {
    n0 = n0_, m0 = m0_, nbox = nbox_, seq0 = seq, issued = 0;
    if (!has_res) return;
    if (lane == 0) bulk_wait_read_all();  // every buffer's last store has read it
    for (; issued < nbox && issued < kBufs; ++issued) issue(issued, lane);
  }
  // Box j's buffer, once its residual has landed (or, without one, once the store that last read
  // the buffer is done with it); null if a wait expired.
  __device__ __forceinline__ __half* acquire(int j, int lane) {
    const int buf = (seq0 + j) % kBufs;
    if (has_res) {
      const int t = j + kBufs - 1;  // refill the buffer of box j - 1 with box t
      if (t < nbox && t == issued) {
        if (lane == 0) bulk_wait_read_all();
        issue(t, lane);
        ++issued;
      }
      if (!mbar_wait_warp(&bar[buf], (phase >> buf) & 1)) return nullptr;
      phase ^= 1u << buf;
      pend &= ~(1u << buf);
    } else {
      if (lane == 0) bulk_wait_read<kBufs - 1>();  // the store of box j - kBufs, the buffer's last user
      __syncwarp();
    }
    return box + buf * 32 * 32;
  }
  // The outputs of box j are in bx: store them.
  __device__ __forceinline__ void store(int j, __half* bx, int lane) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tm_y, bx, n0, m0 + 32 * j);
      bulk_commit_group();
    }
    ++seq;
  }
  // Before the warp exits: every store complete, and no residual copy left in flight (after an
  // expired wait); returns false if draining a copy timed out.
  __device__ __forceinline__ bool finish(int lane) {
    bool ok = true;
    if (lane == 0) {
      bulk_wait_all();
      for (int i = 0; i < kBufs; ++i)
        if (((pend >> i) & 1) && !mbar_wait_bounded(&bar[i], (phase >> i) & 1)) ok = false;
    }
    return ok;
  }
};

}  // namespace wql
