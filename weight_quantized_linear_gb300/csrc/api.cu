// api.cu -- the extern "C" entry points declared in include/wql.h: argument validation, kernel
// selection by shape, launch-error reporting and the per-device error word of bounded waits.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "common.cuh"
#include "internal.h"
#include "trace.cuh"
#include "wql.h"

namespace {

thread_local std::string g_last_error;

// One error word per device (this module's copy on each device that loads the library).
__device__ unsigned g_wql_device_error;

unsigned* device_error_word() {
  static std::atomic<unsigned*> cache[64];  // racing first calls store the same address
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned* w = cache[dev].load(std::memory_order_acquire);
  if (!w) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wql_device_error) != cudaSuccess) return nullptr;
    w = static_cast<unsigned*>(p);
    cache[dev].store(w, std::memory_order_release);
  }
  return w;
}

// One thread waits on an mbarrier that nothing will complete.  The bounded wait gives up after its
// time limit and records kErrTimeoutFull, exactly as a real kernel does when a copy never lands.
__global__ void expire_wait_kernel(unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  wql::mbar_init(&bar, 1);  // one arrival expected, none will come
  wql::fence_mbarrier_init();
  if (!wql::mbar_wait_bounded(&bar, 0)) wql::report_error(err, wql::kErrTimeoutFull);
}

wql_status fail(wql_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

wql_status cuda_status(cudaError_t e, const char* what, const std::string& extra = std::string()) {
  if (e == cudaSuccess) {
    g_last_error.clear();
    return WQL_OK;
  }
  std::string msg = std::string(what) + ": " + cudaGetErrorString(e);
  if (!extra.empty()) msg += " (" + extra + ")";
  return fail(WQL_ECUDA, msg);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define WQL_REQUIRE(cond, msg)                      \
  do {                                              \
    if (!(cond)) return fail(WQL_EINVAL, (msg));    \
  } while (0)

#define WQL_REQUIRE_PTR(p) WQL_REQUIRE((p) != nullptr && aligned16(p), #p " must be a non-null 16-byte aligned device pointer")

bool valid_group(int g) { return g == 32 || g == 64 || g == 128; }

}  // namespace

void wql::set_last_error(const std::string& msg) { g_last_error = msg; }

extern "C" {

const char* wql_status_string(int status) {
  switch (status) {
    case WQL_OK:
      return "ok";
    case WQL_EINVAL:
      return "invalid argument";
    case WQL_EUNSUPPORTED:
      return "unsupported request";
    case WQL_ECUDA:
      return "CUDA error";
    case WQL_ETIMEOUT:
      return "device-side wait timed out";
    default:
      return "unknown status";
  }
}

const char* wql_last_error(void) { return g_last_error.c_str(); }

int wql_version(void) { return 100; }

wql_status wql_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e, "wql_device_status: stream synchronize");
  unsigned* w = device_error_word();
  if (!w) return fail(WQL_ECUDA, "wql_device_status: cannot locate the device error word");
  unsigned v = 0;
  e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e, "wql_device_status: read error word");
  if (v != 0) {
    const unsigned zero = 0;
    cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    char buf[96];
    snprintf(buf, sizeof(buf), "a kernel abandoned a bounded wait (error bits 0x%x)", v);
    return fail(WQL_ETIMEOUT, buf);
  }
  g_last_error.clear();
  return WQL_OK;
}

wql_status wql_awq_pack(const float* w, int K, int N, int group, uint32_t* qweight, uint16_t* scales,
                        uint32_t* qzeros, void* stream) {
  WQL_REQUIRE(valid_group(group), "group must be 32, 64 or 128");
  WQL_REQUIRE(K >= group && K % group == 0, "K must be a positive multiple of the group size");
  WQL_REQUIRE(N >= 32 && N % 32 == 0, "N must be a positive multiple of 32");
  WQL_REQUIRE_PTR(w);
  WQL_REQUIRE_PTR(qweight);
  WQL_REQUIRE_PTR(scales);
  WQL_REQUIRE_PTR(qzeros);
  return cuda_status(wql::launch_awq_pack(w, K, N, group, qweight, scales, qzeros, static_cast<cudaStream_t>(stream)),
                     "wql_awq_pack");
}

namespace {

// wql_w4a16_gemm and wql_w4a16_gemm_silu_mul: one validation and dispatch path.
wql_status w4a16_gemm(const char* fn, const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                      const uint32_t* qzeros, int M, int K, int N, int group, uint16_t* y, int act, void* stream) {
  WQL_REQUIRE(valid_group(group), "group must be 32, 64 or 128");
  WQL_REQUIRE(K >= group && K % group == 0, "K must be a positive multiple of the group size");
  WQL_REQUIRE(N >= 32 && N % 32 == 0, "N must be a positive multiple of 32");
  WQL_REQUIRE(!act || N % 64 == 0, "N must be a multiple of 64 for the gate/up activation");
  WQL_REQUIRE(M >= 0, "M must be >= 0");
  if (M == 0) {
    g_last_error.clear();
    return WQL_OK;
  }
  WQL_REQUIRE_PTR(x);
  WQL_REQUIRE_PTR(qweight);
  WQL_REQUIRE_PTR(scales);
  WQL_REQUIRE_PTR(qzeros);
  WQL_REQUIRE_PTR(y);
  unsigned* dev_err = device_error_word();
  std::string err;
  const char* force = getenv("WQL_FORCE_KERNEL");  // benchmarking switch: "decode" or "prefill"
  const bool prefill = force && strcmp(force, "decode") == 0   ? false
                       : force && strcmp(force, "prefill") == 0 ? true
                                                                : wql::w4a16_use_prefill(M, K, N, group);
  cudaError_t e = prefill ? wql::launch_w4a16_prefill(x, qweight, scales, qzeros, M, K, N, group, y, act, dev_err,
                                                      static_cast<cudaStream_t>(stream), &err)
                          : wql::launch_w4a16_decode(x, qweight, scales, qzeros, M, K, N, group, y, act, dev_err,
                                                     static_cast<cudaStream_t>(stream), &err);
  if (!err.empty()) return fail(WQL_ECUDA, std::string(fn) + ": " + err);
  return cuda_status(e, fn);
}

}  // namespace

wql_status wql_w4a16_gemm(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                          const uint32_t* qzeros, int M, int K, int N, int group, uint16_t* y, void* stream) {
  return w4a16_gemm("wql_w4a16_gemm", x, qweight, scales, qzeros, M, K, N, group, y, 0, stream);
}

wql_status wql_w4a16_gemm_silu_mul(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                                   const uint32_t* qzeros, int M, int K, int N, int group, uint16_t* y,
                                   void* stream) {
  return w4a16_gemm("wql_w4a16_gemm_silu_mul", x, qweight, scales, qzeros, M, K, N, group, y, 1, stream);
}

int wql_w4a16_kernel_for(int M, int K, int N, int group) { return wql::w4a16_use_prefill(M, K, N, group) ? 1 : 0; }

wql_status wql_qrmsnorm_quant_i8(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K, int8_t* q,
                                 float* xs, void* stream) {
  WQL_REQUIRE(K >= 8 && K % 8 == 0, "K must be a positive multiple of 8");
  WQL_REQUIRE(M >= 0, "M must be >= 0");
  if (K > 16384) return fail(WQL_EUNSUPPORTED, "K > 16384 is not supported by the register-resident row kernel");
  if (M == 0) {
    g_last_error.clear();
    return WQL_OK;
  }
  WQL_REQUIRE_PTR(x);
  WQL_REQUIRE_PTR(gamma);
  WQL_REQUIRE_PTR(q);
  WQL_REQUIRE(xs != nullptr && (reinterpret_cast<uintptr_t>(xs) & 3u) == 0, "xs must be a 4-byte aligned device pointer");
  return cuda_status(wql::launch_qrmsnorm_quant_i8(x, gamma, eps, M, K, q, xs, device_error_word(),
                                                   static_cast<cudaStream_t>(stream)),
                     "wql_qrmsnorm_quant_i8");
}

wql_status wql_add_qrmsnorm_quant_i8(const uint16_t* x, const uint16_t* residual, const uint16_t* gamma, float eps,
                                     int M, int K, uint16_t* residual_out, int8_t* q, float* xs, void* stream) {
  WQL_REQUIRE(K >= 8 && K % 8 == 0, "K must be a positive multiple of 8");
  WQL_REQUIRE(M >= 0, "M must be >= 0");
  if (K > 16384) return fail(WQL_EUNSUPPORTED, "K > 16384 is not supported by the register-resident row kernel");
  if (M == 0) {
    g_last_error.clear();
    return WQL_OK;
  }
  WQL_REQUIRE_PTR(x);
  WQL_REQUIRE_PTR(residual);
  WQL_REQUIRE_PTR(gamma);
  WQL_REQUIRE_PTR(residual_out);
  WQL_REQUIRE_PTR(q);
  WQL_REQUIRE(xs != nullptr && (reinterpret_cast<uintptr_t>(xs) & 3u) == 0, "xs must be a 4-byte aligned device pointer");
  return cuda_status(wql::launch_add_qrmsnorm_quant_i8(x, residual, gamma, eps, M, K, residual_out, q, xs,
                                                       device_error_word(), static_cast<cudaStream_t>(stream)),
                     "wql_add_qrmsnorm_quant_i8");
}

namespace {

// Shared argument checks of the QRMSNorm entry points (residual and residual_out only when fused).
wql_status norm_args(const uint16_t* x, const uint16_t* gamma, int M, int K, const void* q, const float* xs,
                     bool fused, const uint16_t* residual, const uint16_t* residual_out) {
  WQL_REQUIRE(K >= 8 && K % 8 == 0, "K must be a positive multiple of 8");
  WQL_REQUIRE(M >= 0, "M must be >= 0");
  if (K > 16384) return fail(WQL_EUNSUPPORTED, "K > 16384 is not supported by the register-resident row kernel");
  if (M == 0) return WQL_OK;
  WQL_REQUIRE_PTR(x);
  WQL_REQUIRE_PTR(gamma);
  WQL_REQUIRE_PTR(q);
  if (fused) {
    WQL_REQUIRE_PTR(residual);
    WQL_REQUIRE_PTR(residual_out);
  }
  WQL_REQUIRE(xs != nullptr && (reinterpret_cast<uintptr_t>(xs) & 3u) == 0, "xs must be a 4-byte aligned device pointer");
  return WQL_OK;
}

}  // namespace

namespace {

wql_status per_token_quant(const char* fn, const uint16_t* x, int M, int K, bool fp8, uint8_t* q, float* xs,
                           void* stream) {
  WQL_REQUIRE(K >= 8 && K % 8 == 0, "K must be a positive multiple of 8");
  WQL_REQUIRE(M >= 0, "M must be >= 0");
  if (K > 16384) return fail(WQL_EUNSUPPORTED, "K > 16384 is not supported by the register-resident row kernel");
  if (M == 0) {
    g_last_error.clear();
    return WQL_OK;
  }
  WQL_REQUIRE_PTR(x);
  WQL_REQUIRE_PTR(q);
  WQL_REQUIRE(xs != nullptr && (reinterpret_cast<uintptr_t>(xs) & 3u) == 0, "xs must be a 4-byte aligned device pointer");
  return cuda_status(wql::launch_per_token_quant(x, M, K, fp8, q, xs, device_error_word(),
                                                 static_cast<cudaStream_t>(stream)),
                     fn);
}

}  // namespace

wql_status wql_per_token_quant_i8(const uint16_t* x, int M, int K, int8_t* q, float* xs, void* stream) {
  return per_token_quant("wql_per_token_quant_i8", x, M, K, false, reinterpret_cast<uint8_t*>(q), xs, stream);
}

wql_status wql_per_token_quant_fp8(const uint16_t* x, int M, int K, uint8_t* q, float* xs, void* stream) {
  return per_token_quant("wql_per_token_quant_fp8", x, M, K, true, q, xs, stream);
}

wql_status wql_qrmsnorm_quant_fp8(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K, uint8_t* q,
                                  float* xs, void* stream) {
  const wql_status st = norm_args(x, gamma, M, K, q, xs, false, nullptr, nullptr);
  if (st != WQL_OK || M == 0) {
    if (st == WQL_OK) g_last_error.clear();
    return st;
  }
  return cuda_status(wql::launch_qrmsnorm_quant_fp8(x, nullptr, gamma, eps, M, K, nullptr, q, xs, device_error_word(),
                                                    static_cast<cudaStream_t>(stream)),
                     "wql_qrmsnorm_quant_fp8");
}

wql_status wql_add_qrmsnorm_quant_fp8(const uint16_t* x, const uint16_t* residual, const uint16_t* gamma, float eps,
                                      int M, int K, uint16_t* residual_out, uint8_t* q, float* xs, void* stream) {
  const wql_status st = norm_args(x, gamma, M, K, q, xs, true, residual, residual_out);
  if (st != WQL_OK || M == 0) {
    if (st == WQL_OK) g_last_error.clear();
    return st;
  }
  return cuda_status(wql::launch_qrmsnorm_quant_fp8(x, residual, gamma, eps, M, K, residual_out, q, xs,
                                                    device_error_word(), static_cast<cudaStream_t>(stream)),
                     "wql_add_qrmsnorm_quant_fp8");
}

size_t wql_w8a8_workspace_bytes(int M, int K, int N) {
  (void)N;
  if (M < wql::kW8A8PrefillMinM || K <= 0) return 0;  // the streaming decode kernel needs no scratch
  return wql::w8a8_prefill_workspace_bytes(M, K);      // fp16 copy of the activation codes
}

namespace {

// wql_w8a8_gemm and wql_w8a8_gemm_fused: one validation and dispatch path.
wql_status w8a8_gemm(const char* fn, const int8_t* q, const float* xs, const int8_t* qw, const float* ws,
                     const uint16_t* bias, const uint16_t* residual, int M, int K, int N, uint16_t* y,
                     int32_t* acc_out, void* workspace, size_t workspace_bytes, void* stream) {
  WQL_REQUIRE(K >= 16 && K % 16 == 0, "K must be a positive multiple of 16");
  WQL_REQUIRE(K <= 131072, "K must be <= 131072 so that the int32 accumulator cannot overflow");
  WQL_REQUIRE(N >= 32 && N % 32 == 0, "N must be a positive multiple of 32");
  WQL_REQUIRE(M >= 0, "M must be >= 0");
  if (M == 0) {
    g_last_error.clear();
    return WQL_OK;
  }
  WQL_REQUIRE_PTR(q);
  WQL_REQUIRE_PTR(qw);
  WQL_REQUIRE_PTR(ws);
  WQL_REQUIRE_PTR(y);
  WQL_REQUIRE(xs != nullptr && (reinterpret_cast<uintptr_t>(xs) & 3u) == 0, "xs must be a 4-byte aligned device pointer");
  WQL_REQUIRE(acc_out == nullptr || aligned16(acc_out), "acc_out must be NULL or 16-byte aligned");
  WQL_REQUIRE(bias == nullptr || aligned16(bias), "bias must be NULL or 16-byte aligned");
  WQL_REQUIRE(residual == nullptr || aligned16(residual), "residual must be NULL or 16-byte aligned");
  const size_t need = wql_w8a8_workspace_bytes(M, K, N);
  WQL_REQUIRE(workspace_bytes >= need, "workspace is smaller than wql_w8a8_workspace_bytes()");
  WQL_REQUIRE(need == 0 || (workspace != nullptr && aligned16(workspace)), "workspace must be 16-byte aligned");
  unsigned* dev_err = device_error_word();
  std::string err;
  const char* force = getenv("WQL_FORCE_KERNEL");  // benchmarking switch: "decode" or "prefill"
  const bool prefill = force && strcmp(force, "decode") == 0 ? false : M >= wql::kW8A8PrefillMinM;
  cudaError_t e = prefill ? wql::launch_w8a8_prefill(q, xs, qw, ws, M, K, N, y, acc_out, bias, residual, workspace,
                                                     dev_err, static_cast<cudaStream_t>(stream), &err)
                          : wql::launch_w8a8_decode(q, xs, qw, ws, M, K, N, y, acc_out, bias, residual, dev_err,
                                                    static_cast<cudaStream_t>(stream), &err);
  if (!err.empty()) return fail(WQL_ECUDA, std::string(fn) + ": " + err);
  return cuda_status(e, fn);
}

}  // namespace

wql_status wql_w8a8_gemm(const int8_t* q, const float* xs, const int8_t* qw, const float* ws, int M, int K, int N,
                         uint16_t* y, int32_t* acc_out, void* workspace, size_t workspace_bytes, void* stream) {
  return w8a8_gemm("wql_w8a8_gemm", q, xs, qw, ws, nullptr, nullptr, M, K, N, y, acc_out, workspace,
                   workspace_bytes, stream);
}

wql_status wql_w8a8_gemm_fused(const int8_t* q, const float* xs, const int8_t* qw, const float* ws,
                               const uint16_t* bias, const uint16_t* residual, int M, int K, int N, uint16_t* y,
                               int32_t* acc_out, void* workspace, size_t workspace_bytes, void* stream) {
  return w8a8_gemm("wql_w8a8_gemm_fused", q, xs, qw, ws, bias, residual, M, K, N, y, acc_out, workspace,
                   workspace_bytes, stream);
}

wql_status wql_w8a8_gemm_fp8(const uint8_t* q, const float* xs, const uint8_t* qw, const float* ws,
                             const uint16_t* bias, const uint16_t* residual, int M, int K, int N, uint16_t* y,
                             float* acc_out, void* stream) {
  WQL_REQUIRE(K >= 16 && K % 16 == 0, "K must be a positive multiple of 16");
  WQL_REQUIRE(N >= 32 && N % 32 == 0, "N must be a positive multiple of 32");
  WQL_REQUIRE(M >= 0, "M must be >= 0");
  if (M == 0) {
    g_last_error.clear();
    return WQL_OK;
  }
  WQL_REQUIRE_PTR(q);
  WQL_REQUIRE_PTR(qw);
  WQL_REQUIRE_PTR(ws);
  WQL_REQUIRE_PTR(y);
  WQL_REQUIRE(xs != nullptr && (reinterpret_cast<uintptr_t>(xs) & 3u) == 0, "xs must be a 4-byte aligned device pointer");
  WQL_REQUIRE(acc_out == nullptr || aligned16(acc_out), "acc_out must be NULL or 16-byte aligned");
  WQL_REQUIRE(bias == nullptr || aligned16(bias), "bias must be NULL or 16-byte aligned");
  WQL_REQUIRE(residual == nullptr || aligned16(residual), "residual must be NULL or 16-byte aligned");
  unsigned* dev_err = device_error_word();
  std::string err;
  const char* force = getenv("WQL_FORCE_KERNEL");  // benchmarking switch: "decode"
  const bool prefill = force && strcmp(force, "decode") == 0 ? false : M >= wql::kFp8PrefillMinM;
  cudaError_t e = prefill ? wql::launch_fp8_prefill(q, xs, qw, ws, M, K, N, y, acc_out, bias, residual, dev_err,
                                                    static_cast<cudaStream_t>(stream), &err)
                          : wql::launch_fp8_decode(q, xs, qw, ws, M, K, N, y, acc_out, bias, residual, dev_err,
                                                   static_cast<cudaStream_t>(stream), &err);
  if (!err.empty()) return fail(WQL_ECUDA, "wql_w8a8_gemm_fp8: " + err);
  return cuda_status(e, "wql_w8a8_gemm_fp8");
}

wql_status wql_act_absmax(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K, float* absmax,
                          void* stream) {
  WQL_REQUIRE(K >= 8 && K % 8 == 0, "K must be a positive multiple of 8");
  WQL_REQUIRE(M >= 0, "M must be >= 0");
  if (K > 16384) return fail(WQL_EUNSUPPORTED, "K > 16384 is not supported by the register-resident row kernel");
  WQL_REQUIRE_PTR(absmax);
  if (M > 0) {
    WQL_REQUIRE_PTR(x);
    WQL_REQUIRE_PTR(gamma);
  }
  return cuda_status(wql::launch_act_absmax(x, gamma, eps, M, K, absmax, device_error_word(),
                                            static_cast<cudaStream_t>(stream)),
                     "wql_act_absmax");
}

wql_status wql_smooth(const float* absmax, const uint16_t* gamma, const float* w, int K, int N, float* s,
                      uint16_t* gamma_out, float* w_out, void* stream) {
  WQL_REQUIRE(K >= 16 && K % 16 == 0, "K must be a positive multiple of 16");
  WQL_REQUIRE(N >= 32 && N % 32 == 0, "N must be a positive multiple of 32");
  WQL_REQUIRE_PTR(absmax);
  WQL_REQUIRE_PTR(gamma);
  WQL_REQUIRE_PTR(w);
  WQL_REQUIRE_PTR(s);
  WQL_REQUIRE_PTR(gamma_out);
  WQL_REQUIRE_PTR(w_out);
  return cuda_status(wql::launch_smooth(absmax, gamma, w, K, N, s, gamma_out, w_out, static_cast<cudaStream_t>(stream)),
                     "wql_smooth");
}

wql_status wql_per_channel_quant_i8(const float* w, int K, int N, int8_t* qw, float* ws, void* stream) {
  WQL_REQUIRE(K >= 16 && K % 16 == 0, "K must be a positive multiple of 16");
  WQL_REQUIRE(N >= 32 && N % 32 == 0, "N must be a positive multiple of 32");
  WQL_REQUIRE_PTR(w);
  WQL_REQUIRE_PTR(qw);
  WQL_REQUIRE_PTR(ws);
  return cuda_status(wql::launch_per_channel_quant_i8(w, K, N, qw, ws, static_cast<cudaStream_t>(stream)),
                     "wql_per_channel_quant_i8");
}

wql_status wql_per_channel_quant_fp8(const float* w, int K, int N, uint8_t* qw, float* ws, void* stream) {
  WQL_REQUIRE(K >= 16 && K % 16 == 0, "K must be a positive multiple of 16");
  WQL_REQUIRE(N >= 32 && N % 32 == 0, "N must be a positive multiple of 32");
  WQL_REQUIRE_PTR(w);
  WQL_REQUIRE_PTR(qw);
  WQL_REQUIRE_PTR(ws);
  return cuda_status(wql::launch_per_channel_quant_fp8(w, K, N, qw, ws, static_cast<cudaStream_t>(stream)),
                     "wql_per_channel_quant_fp8");
}

wql_status wql_kv_quant_i8(const uint16_t* kv, int64_t rows, int D, int8_t* q, float* scales, void* stream) {
  WQL_REQUIRE(D >= 128 && D % 128 == 0, "D must be a positive multiple of 128");
  WQL_REQUIRE(rows >= 0, "rows must be >= 0");
  if (rows == 0) {
    g_last_error.clear();
    return WQL_OK;
  }
  WQL_REQUIRE_PTR(kv);
  WQL_REQUIRE_PTR(q);
  WQL_REQUIRE(scales != nullptr && (reinterpret_cast<uintptr_t>(scales) & 3u) == 0,
              "scales must be a 4-byte aligned device pointer");
  return cuda_status(wql::launch_kv_quant_i8(kv, rows, D, q, scales, static_cast<cudaStream_t>(stream)),
                     "wql_kv_quant_i8");
}

wql_status wql_kv_dequant_i8(const int8_t* q, const float* scales, int64_t rows, int D, uint16_t* out, void* stream) {
  WQL_REQUIRE(D >= 128 && D % 128 == 0, "D must be a positive multiple of 128");
  WQL_REQUIRE(rows >= 0, "rows must be >= 0");
  if (rows == 0) {
    g_last_error.clear();
    return WQL_OK;
  }
  WQL_REQUIRE_PTR(q);
  WQL_REQUIRE_PTR(out);
  WQL_REQUIRE(scales != nullptr && (reinterpret_cast<uintptr_t>(scales) & 3u) == 0,
              "scales must be a 4-byte aligned device pointer");
  return cuda_status(wql::launch_kv_dequant_i8(q, scales, rows, D, out, static_cast<cudaStream_t>(stream)),
                     "wql_kv_dequant_i8");
}

wql_status wql_diag_expire_wait(void* stream) {
  unsigned* dev_err = device_error_word();
  if (!dev_err) return fail(WQL_ECUDA, "wql_diag_expire_wait: cannot locate the device error word");
  expire_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(dev_err);
  return cuda_status(cudaGetLastError(), "wql_diag_expire_wait");
}

wql_status wql_trace_setup(uint64_t* buf, const void* ybase, uint64_t ystride, int launches, int ctas) {
#ifdef WQL_PHASE_TRACE
  WQL_REQUIRE(buf == nullptr || (launches > 0 && ctas > 0 && ystride > 0 &&
                                 (reinterpret_cast<uintptr_t>(buf) & 7u) == 0),
              "buf must be null, or 8-byte aligned with positive launches, ctas and ystride");
  wql::TraceDesc d{reinterpret_cast<unsigned long long*>(buf), reinterpret_cast<unsigned long long>(ybase),
                   (unsigned long long)ystride, launches, ctas};
  cudaError_t e = wql::trace_set_w4a16_decode(d);
  if (e == cudaSuccess) e = wql::trace_set_w4a16_prefill(d);
  return cuda_status(e, "wql_trace_setup");
#else
  (void)buf;
  (void)ybase;
  (void)ystride;
  (void)launches;
  (void)ctas;
  return fail(WQL_EUNSUPPORTED, "wql_trace_setup: this library was built without WQL_PHASE_TRACE");
#endif
}

}  // extern "C"
