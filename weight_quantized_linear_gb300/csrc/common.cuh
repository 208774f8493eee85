// common.cuh -- device helpers shared by the sm_103a kernels of libwql.so:
// mbarrier / TMA / cluster primitives as inline PTX, bounded waits, the device error word.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace wql {

// Bits of the device-side error word (one 32-bit word per device, owned by api.cu and passed to
// every kernel that can abandon a wait).
enum : unsigned {
  kErrTimeoutFull = 1u,    // consumer gave up waiting for a TMA stage
  kErrTimeoutEmpty = 2u,   // producer gave up waiting for a free stage
  kErrTimeoutMma = 4u,     // MMA / accumulator hand-off wait expired
  kErrTimeoutDrain = 8u,   // exit-time drain of in-flight copies expired
  kErrSmemAlign = 16u,     // dynamic shared memory not 1024-byte aligned where a kernel has no slack for it
};

// A bounded wait polls for at most this long (nanoseconds of %globaltimer).  Normal waits take
// microseconds; 2 s means something is broken, and the kernel then records an error and exits.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------------------------
// mbarrier (shared::cta)
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false if the limit expired.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ void report_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

// ---------------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), tensor maps passed as __grid_constant__ kernel parameters
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2D tiled load of the box at (x = inner coordinate, y = outer coordinate) into shared memory;
// completion is signalled on `bar` as transaction bytes.  x * element size must be a multiple
// of 16 bytes (callers only pass multiples of the box width).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Same with an L2 eviction-priority hint (policy from createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                                 int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2D tiled store of a shared-memory box to global memory at (x = inner, y = outer coordinate); the
// part of the box outside the tensor is not written.  Completion is tracked per issuing thread
// through bulk groups: bulk_commit_group() after the stores, then one of the waits below.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* smem_src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Every bulk store committed by this thread has finished reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// All but the newest N bulk store groups committed by this thread have finished reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Every bulk store committed by this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Generic-proxy writes to shared memory become visible to the async proxy (tensor cores, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------------------------
// Thread-block clusters
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Split cluster barrier: a relaxed arrival at kernel start, and the matching wait just before the
// first access to a peer's shared memory (which must not happen before every peer has started).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_cluster_i4(uint32_t addr, int4 v) {
  asm volatile("st.shared::cluster.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Asynchronous store of 16 bytes into a peer CTA's shared memory; its completion is counted as 16
// transaction bytes on the peer's mbarrier (both addresses in the shared::cluster window).
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from this CTA's shared
// memory to the shared memory of a CTA of the cluster; completes transaction bytes on that CTA's
// mbarrier.  Both remote addresses come from mapa.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t remote_dst, uint32_t local_src, uint32_t bytes,
                                                  uint32_t remote_bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   remote_dst),
               "r"(local_src), "r"(bytes), "r"(remote_bar)
               : "memory");
}

__device__ __forceinline__ void st_async_f4(uint32_t remote_addr, float4 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   remote_addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
               : "memory");
}

__device__ __forceinline__ void st_async_i4(uint32_t remote_addr, int4 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.s32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   remote_addr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
               : "memory");
}

// 3D tiled TMA load (coordinates x innermost).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Owner rank of float4 index f when nq float4s are split into `parts` contiguous slices
// [floor(nq r / parts), floor(nq (r + 1) / parts)).
__device__ __forceinline__ int slice_owner(int f, int nq, int parts) {
  int r = (int)(((long long)f * parts) / nq);
  while (r + 1 < parts && (int)((long long)nq * (r + 1) / parts) <= f) ++r;
  while (r > 0 && (int)((long long)nq * r / parts) > f) --r;
  return r;
}

// shared::cta address -> the same offset in CTA `rank` of this cluster (shared::cluster window).
__device__ __forceinline__ uint32_t map_cluster_addr(uint32_t smem_addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr), "r"(rank));
  return out;
}

// Address of the same shared-memory variable in CTA `rank` of this cluster (shared::cluster).
__device__ __forceinline__ uint32_t map_cluster(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  // volatile keeps these loads after the cluster barrier; no memory clobber, so several can be in
  // flight before their values are used
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ int4 ld_cluster_i4(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared::cluster.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Named barrier over `count` threads (a multiple of 32) of this CTA; id 0 is __syncthreads.
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------------------------
// Programmatic dependent launch: wait until the preceding kernel's writes are visible.
// A no-op when the launch did not use the programmatic-serialization attribute.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------------------------
// Small bit helpers
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & mask) | bits, as one LOP3
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t bits) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));
  return d;
}

__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---------------------------------------------------------------------------------------------
// int8 codes of per-row / per-group symmetric quantisation (s = absmax / 127)
// ---------------------------------------------------------------------------------------------

// Round to the nearest integer (ties to even) and saturate to [-128, 127], in one conversion.
__device__ __forceinline__ int cvt_rni_sat_s8(float f) {
  int r;
  asm("{\n .reg .s8 t;\n cvt.rni.sat.s8.f32 t, %1;\n cvt.s32.s8 %0, t;\n}" : "=r"(r) : "f"(f));
  return r;
}

// clamp(round_half_even(fl(y / s)), -128, 127), without a division in the common case.
// t = fl(y * inv) with inv = fl(1 / s) lies within 2.3e-5 of fl(y / s) when |y / s| <= 127.5
// (two roundings of relative size 2^-24 each, plus fl(y / s)'s own half ulp), so whenever t is
// more than 5e-5 from a half-integer (|t - rint(t)| < 0.49995), both round to the same integer.
// quant_fast returns rint(t) saturated and sets `exact` when that is not guaranteed; quant_exact
// then divides.
__device__ __forceinline__ int quant_fast(float y, float inv, bool& exact) {
  const float t = __fmul_rn(y, inv);
  const float rt = rintf(t);
  exact |= !(fabsf(__fsub_rn(t, rt)) < 0.49995f);
  return cvt_rni_sat_s8(rt);
}
__device__ __forceinline__ int quant_exact(float y, float s, float inv) {
  const float t = __fmul_rn(y, inv);
  const float rt = rintf(t);
  if (fabsf(__fsub_rn(t, rt)) < 0.49995f) return cvt_rni_sat_s8(rt);
  return cvt_rni_sat_s8(__fdiv_rn(y, s));
}

// ---------------------------------------------------------------------------------------------
// float8 e4m3 ("fn": finite only, largest value 448)
// ---------------------------------------------------------------------------------------------

// Four fp32 -> four e4m3 bytes (a0 in byte 0), nearest value with ties to even, magnitudes beyond
// 448 saturated to 448.
__device__ __forceinline__ uint32_t e4m3x4_rn_sat(float a0, float a1, float a2, float a3) {
  uint32_t r;
  asm("{\n .reg .b16 lo, hi;\n"
      " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
      " mov.b32 %0, {lo, hi};\n}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return r;
}

// e4m3 codes of fl(y_i / s) for four values, without a division in the common case.
// t = fl(y * inv) with inv = fl(1 / s) lies within 3 fp32 ulps of fl(y / s) (two roundings of
// relative size 2^-24 and fl(y / s)'s own half ulp).  Rounding to e4m3 is monotonic, so when the
// values 8 ulps below and above t (one step of the bit pattern is one ulp) give the same codes,
// every value between them does, fl(y / s) included.  Otherwise -- near an e4m3 rounding tie, or
// at zero, where a step below wraps to NaN -- the codes come from the correctly rounded quotient.
__device__ __forceinline__ uint32_t e4m3x4_div(const float (&y)[4], float s, float inv) {
  float lo[4], hi[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b = __float_as_int(__fmul_rn(y[i], inv));
    lo[i] = __int_as_float(b - 8);
    hi[i] = __int_as_float(b + 8);
  }
  const uint32_t a = e4m3x4_rn_sat(lo[0], lo[1], lo[2], lo[3]);
  if (a == e4m3x4_rn_sat(hi[0], hi[1], hi[2], hi[3])) return a;
  return e4m3x4_rn_sat(__fdiv_rn(y[0], s), __fdiv_rn(y[1], s), __fdiv_rn(y[2], s), __fdiv_rn(y[3], s));
}

// Four e4m3 bytes -> two f16x2 (bytes 0,1 and bytes 2,3), exact: every e4m3 value is an fp16 value.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t v, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n"
      " mov.b32 {a, b}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n"
      " cvt.rn.f16x2.e4m3x2 %1, b;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(v));
}

// The activation of a fused gate/up projection ("FastLLM architecture" article, section 2): from the
// GEMM's fp32 gate and up values g and u of one output, fp16(silu(g16) * u16) with g16, u16 the fp16
// outputs the unfused GEMM would have written and silu(g) = g / (1 + exp(-g)) in fp32 (IEEE
// division; expf as the CUDA math library provides it).
__device__ __forceinline__ __half silu_mul_h(float g, float u) {
  const float g16 = __half2float(__float2half_rn(g)), u16 = __half2float(__float2half_rn(u));
  const float sg = __fdiv_rn(g16, __fadd_rn(1.0f, expf(-g16)));
  return __float2half_rn(__fmul_rn(sg, u16));
}

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_f16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Transposed: lane 4g + t receives b16 column g of rows 2t and 2t + 1 of each 8 x 8 matrix.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint2 lds_u64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds_u128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

}  // namespace wql
