// internal.h -- host-side declarations shared by the translation units of libwql.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace wql {

// Encode a 2D tiled TMA descriptor for a row-major matrix [outer, inner] of `elem_bytes`-sized
// elements with a row pitch of `row_bytes`.  Returns false and fills *err on failure.
bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base,
                  uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swizzle, std::string* err);

// Encode a 3D tiled TMA descriptor: element (x, y, z) at base + x*elem + y*stride1 + z*stride2.
bool make_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2,
                  CUtensorMapSwizzle swizzle, std::string* err);

int num_sms();  // SM count of the current device (cached per device)

// Sets the message returned by wql_last_error() on this host thread.
void set_last_error(const std::string& msg);

// Split factor S (cluster size along k, 1..8) for a split-K launch of `units` independent output
// tiles: the largest S whose units * S CTAs are all co-resident in one wave (occupancy query with
// the cluster attribute, cached per kernel and device), bounded by the number of k blocks.  With
// `pow2`, S is restricted to powers of two.  With `balanced`, S instead minimises the load of the
// busiest SM (several co-resident CTAs per SM and several rounds allowed).  The kernel is queried
// with a (1, S, 1) cluster.
int pick_k_split(const void* kernel, int threads, int smem_bytes, int units, int kblocks, bool pow2 = false,
                 bool balanced = false);

// Launchers.  Each returns cudaSuccess or the launch error; *err gets a message for
// non-CUDA failures (descriptor encoding).  Arguments are already validated by api.cu.
cudaError_t launch_awq_pack(const float* w, int K, int N, int group, uint32_t* qweight,
                            uint16_t* scales, uint32_t* qzeros, cudaStream_t s);

// act = 0: y [M, N]; act = 1: the gate/up activation, y [M, N / 2] with y[m, j] =
// fp16(silu(fp16(y2[m, 2j])) * fp16(y2[m, 2j + 1])) of the GEMM's output y2.
cudaError_t launch_w4a16_decode(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                                const uint32_t* qzeros, int M, int K, int N, int group, uint16_t* y, int act,
                                unsigned* dev_err, cudaStream_t s, std::string* err);

cudaError_t launch_w4a16_prefill(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                                 const uint32_t* qzeros, int M, int K, int N, int group, uint16_t* y, int act,
                                 unsigned* dev_err, cudaStream_t s, std::string* err);

// Token count from which w4a16_gemm always uses the tcgen05 kernel instead of the streaming decode
// kernel; from 17 tokens on it does so for the shapes w4a16_use_prefill picks.
constexpr int kW4A16PrefillMinM = 33;

// Kernel choice for w4a16_gemm.  Up to 16 tokens the decode kernel streams each weight tile once.
// From 17 to 32 it runs two 16-token blocks, so every tile is dequantised twice, and its per-group
// epilogue runs once per 128 k at G = 128 but four times at G = 32.  The tcgen05 kernel (one
// 32-token tile) is then faster when its output tiles of 128 channels fill most SMs in one wave,
// when K is long enough for its split-K, at G = 32 for every shape, and at G = 64 also beyond one
// wave (measured on GB300, us, decode vs tcgen05 at M = 32, K = 4096 unless stated):
//   G = 128: N = 4096 7.8 / 9.3, N = 12288 22.8 / 18.5, N = 22016 27.9 / 31.7, K = 11008 17.8 / 16.4;
//   G = 64:  N = 4096 7.7 / 9.5, N = 12288 24.9 / 16.4, N = 22016 36.5 / 30.8, K = 11008 17.8 / 15.6;
//   G = 32:  N = 4096 10.6 / 9.8, N = 12288 31.6 / 17.0, N = 22016 53.4 / 33.4, K = 11008 24.4 / 16.1.
inline bool w4a16_use_prefill(int M, int K, int N, int group) {
  if (M >= kW4A16PrefillMinM) return true;
  if (M <= 16) return false;
  const int ntn = (N + 127) / 128, sms = num_sms();
  if (K >= 8192 || group == 32) return true;
  if (2 * ntn < sms) return false;
  return ntn <= sms || group < 128;
}

cudaError_t launch_qrmsnorm_quant_i8(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K,
                                     int8_t* q, float* xs, unsigned* dev_err, cudaStream_t s);

cudaError_t launch_add_qrmsnorm_quant_i8(const uint16_t* x, const uint16_t* residual, const uint16_t* gamma,
                                         float eps, int M, int K, uint16_t* residual_out, int8_t* q, float* xs,
                                         unsigned* dev_err, cudaStream_t s);

// per_token_quant of plain fp16 rows: xs = absmax / 127 (int8) or / 448 (fp8), q the codes of x / xs.
cudaError_t launch_per_token_quant(const uint16_t* x, int M, int K, bool fp8, uint8_t* q, float* xs, unsigned* dev_err,
                                   cudaStream_t s);

cudaError_t launch_act_absmax(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K,
                              float* absmax, unsigned* dev_err, cudaStream_t s);

cudaError_t launch_smooth(const float* absmax, const uint16_t* gamma, const float* w, int K, int N,
                          float* s_out, uint16_t* gamma_out, float* w_out, cudaStream_t s);

cudaError_t launch_per_channel_quant_i8(const float* w, int K, int N, int8_t* qw, float* ws,
                                        cudaStream_t s);

// Token count from which w8a8_gemm uses the tcgen05 kernel (which needs the workspace).
constexpr int kW8A8PrefillMinM = 17;
size_t w8a8_prefill_workspace_bytes(int M, int K);
// bias [N] and residual [M, N] (fp16, either may be null) are the optional epilogue terms
// y = fp16(((acc * xs) * ws + bias) + residual).
cudaError_t launch_w8a8_prefill(const int8_t* q, const float* xs, const int8_t* qw, const float* ws, int M, int K,
                                int N, uint16_t* y, int32_t* acc_out, const uint16_t* bias, const uint16_t* residual,
                                void* workspace, unsigned* dev_err, cudaStream_t stream, std::string* err);

cudaError_t launch_w8a8_decode(const int8_t* q, const float* xs, const int8_t* qw, const float* ws,
                               int M, int K, int N, uint16_t* y, int32_t* acc_out, const uint16_t* bias,
                               const uint16_t* residual, unsigned* dev_err, cudaStream_t s, std::string* err);

// fp8 (e4m3) variant.  residual (and residual_out) may be null: then the plain QRMSNorm.
cudaError_t launch_qrmsnorm_quant_fp8(const uint16_t* x, const uint16_t* residual, const uint16_t* gamma, float eps,
                                      int M, int K, uint16_t* residual_out, uint8_t* q, float* xs, unsigned* dev_err,
                                      cudaStream_t s);

cudaError_t launch_per_channel_quant_fp8(const float* w, int K, int N, uint8_t* qw, float* ws, cudaStream_t s);

// Token count from which the fp8 GEMM uses the tcgen05 kernel; below it, the streaming decode kernel.
constexpr int kFp8PrefillMinM = 17;
int fp8_prefill_tile_n(int M, int N);
cudaError_t launch_fp8_prefill(const uint8_t* q, const float* xs, const uint8_t* qw, const float* ws, int M, int K,
                               int N, uint16_t* y, float* acc_out, const uint16_t* bias, const uint16_t* residual,
                               unsigned* dev_err, cudaStream_t stream, std::string* err);
cudaError_t launch_fp8_decode(const uint8_t* q, const float* xs, const uint8_t* qw, const float* ws, int M, int K,
                              int N, uint16_t* y, float* acc_out, const uint16_t* bias, const uint16_t* residual,
                              unsigned* dev_err, cudaStream_t stream, std::string* err);

// KV cache int8 in groups of 128 channels: kv [rows, D] fp16, D % 128 == 0.
cudaError_t launch_kv_quant_i8(const uint16_t* kv, long long rows, int D, int8_t* q, float* scales, cudaStream_t s);
cudaError_t launch_kv_dequant_i8(const int8_t* q, const float* scales, long long rows, int D, uint16_t* out,
                                 cudaStream_t s);

#ifdef WQL_PHASE_TRACE
// Phase-trace builds only: register the stamp buffer with the traced kernels of each source file.
struct TraceDesc;
cudaError_t trace_set_w4a16_decode(const TraceDesc& d);
cudaError_t trace_set_w4a16_prefill(const TraceDesc& d);
#endif

}  // namespace wql
