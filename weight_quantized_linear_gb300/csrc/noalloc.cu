// noalloc.cu -- wql_w8a8_gemm_noalloc: the int8 GEMM for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory at call time: an inference engine that hands
// its whole device memory budget to its own pool (KV cache, activations) up front, a plugin hosted
// by a framework that owns every allocation and forbids its plugins from calling cudaMalloc, or a
// latency-critical loop that must not pay for the allocator's implicit device synchronisation.
// wql_w8a8_gemm needs a workspace of M*K*2 bytes for its tensor-core path (an fp16 copy of the
// activation codes); this entry point uses a fixed scratch array compiled into the library instead
// and otherwise runs exactly the same kernels.
#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"
#include "wql.h"

namespace {

// Fixed scratch for the fp16 copy of the activation codes and their row-norm maxima: 32 MiB +
// 64 KiB, i.e. M * K * 2 + 16384 bytes up to M = K = 4096.  It exists once per GPU that loads the library
// and lives until the process exits.
constexpr size_t kScratchBytes = (size_t(32) << 20) + (size_t(64) << 10);
static __device__ __align__(256) unsigned char g_w8a8_scratch[kScratchBytes];

// The array's device address, looked up once per device (with that device current).  Host code must
// never pass `g_w8a8_scratch` itself: on the host that name is only a stand-in for the device symbol.
void* scratch_address(std::string* err) {
  static std::mutex mu;
  static void* cache[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *err = std::string("cannot determine the current device: ") + cudaGetErrorString(e);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_w8a8_scratch);
    if (e != cudaSuccess || p == nullptr) {
      *err = std::string("cudaGetSymbolAddress of the static scratch failed: ") + cudaGetErrorString(e);
      return nullptr;
    }
    cache[dev] = p;
  }
  return cache[dev];
}

}  // namespace

extern "C" {

wql_status wql_w8a8_gemm_noalloc(const int8_t* q, const float* xs, const int8_t* qw, const float* ws, int M, int K,
                                 int N, uint16_t* y, int32_t* acc_out, void* stream) {
  const size_t need = (M > 0 && K > 0 && N > 0) ? wql_w8a8_workspace_bytes(M, K, N) : 0;
  if (need > kScratchBytes) {
    wql::set_last_error("wql_w8a8_gemm_noalloc: this call needs " + std::to_string(need) +
                        " bytes of scratch (M * K * 2 + 16384) but the static scratch holds " + std::to_string(kScratchBytes) +
                        " bytes; use wql_w8a8_gemm with a caller-provided workspace");
    return WQL_EUNSUPPORTED;
  }
  void* scratch = nullptr;
  if (need > 0) {
    std::string err;
    scratch = scratch_address(&err);
    if (!scratch) {
      wql::set_last_error("wql_w8a8_gemm_noalloc: " + err);
      return WQL_ECUDA;
    }
  }
  // Same validation, kernels and results as wql_w8a8_gemm; the pre-pass overwrites every scratch
  // byte it later reads, so nothing left over from an earlier call is ever used.
  return wql_w8a8_gemm(q, xs, qw, ws, M, K, N, y, acc_out, scratch, need > 0 ? kScratchBytes : 0, stream);
}

}  // extern "C"
