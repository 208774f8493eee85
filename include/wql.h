/*
 * wql.h -- C ABI of the GB300 (sm_103a) weight-quantized linear library (libwql.so).
 *
 * Two quantized linear layers as used by LLM serving engines:
 *   - AWQ-format W4A16: int4 weights packed 8 per uint32, one fp16 scale and one 4-bit zero
 *     point per group of 32/64/128 input channels, fp16 activations and output.
 *   - SmoothQuant W8A8: RMSNorm fused with per-token dynamic int8 quantisation, then an
 *     int8 x int8 -> int32 GEMM dequantised by per-token x per-channel scales.
 *
 * Sources (titles of the public write-ups the operations follow):
 *   [AWQ]  "LMDeploy ... INT4 quantisation" tutorial, section 2: AWQ quantises weights per group
 *          with an asymmetric zero point from each group's own min/max; group sizes 32/64/128.
 *   [TM]   same tutorial, section 5.1: the fp16 x int4 GEMM kernel of the serving engine.
 *   [AUQ]  "AUQ dual-process framework" article, section 3.3 (per-group scale and zero point)
 *          and section 5.4 (checkpoint tensors qweight, scales, zeros; dim 0 of qweight is the
 *          grouped input dimension, a multiple of 128 for group 128).
 *   [W8A8] "LMDeploy W8A8 quantisation guide": weight smoothing (smooth_ln_fcs, alpha 0.5),
 *          QRMSNorm / QLinear modules, per_token_quant_int8 (scale = absmax / 127),
 *          per_channel_quant (fp32 scale per output channel), matmul_kernel_dynamic_quant
 *          (int32 accumulator, c = c * rms_scale * linear_scale), and its fp8 variant.
 *   [FastLLM] "FastLLM architecture" article, section 5.2: KV cache int8 in groups of 128.
 *
 * Conventions for every entry point:
 *   - Matrices are row-major and dense (no strides).  K = input features, N = output
 *     features, M = tokens (rows of the activation), G = group size.
 *   - fp16 data is passed as uint16_t bit patterns (IEEE binary16).
 *   - Every pointer is DEVICE memory owned by the caller, 16-byte aligned.  The library never
 *     allocates, frees or keeps a pointer after the call returns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only enqueue work
 *     on that stream and return; outputs are valid once the stream reaches that point.
 *   - Arguments are validated before anything is enqueued.  On WQL_EINVAL / WQL_EUNSUPPORTED
 *     nothing is launched and outputs are untouched; wql_last_error() describes the problem.
 *     WQL_ECUDA reports a launch failure (cudaGetLastError after the launch).
 *   - Kernels that wait on on-chip barriers give up after a bounded time instead of hanging;
 *     they then record a device-side error that wql_device_status() returns as WQL_ETIMEOUT.
 *   - M = 0 is a valid empty call: it returns WQL_OK and launches nothing.
 *   - The library holds no per-call state; calls on different streams may run concurrently.
 *     It keeps per-device state for the life of the process (kernel attributes, the device
 *     error word's address, the scratch-free GEMM's array address).  cudaDeviceReset
 *     invalidates that state: no call may follow a reset of that device in the same process.
 *   - Weight prefetch (programmatic dependent launch): the W4A16 GEMMs and the decode path of the
 *     W8A8 GEMMs (int8 and fp8, up to 16 tokens) are launched so that they may start while the
 *     kernel enqueued just before them on the stream is still running, and they begin copying
 *     their WEIGHT operands (qweight / scales / qzeros, or qw) before that kernel has finished;
 *     only the activations and the outputs wait for it.  So the weight buffers must already
 *     hold their final contents when the preceding kernel on the stream starts finishing:
 *       * the library's own weight writers (wql_awq_pack, wql_per_channel_quant_i8/_fp8) make
 *         their writes visible device-wide before they exit, so pack-then-GEMM on one stream
 *         with nothing in between is safe;
 *       * a caller's kernel that writes weight buffers and is enqueued directly before one of
 *         these GEMMs must end each thread's writes with a device-scope fence (__threadfence()),
 *         or the two must be separated by something that is not a kernel launch (an event
 *         record/wait, a memcpy, a stream synchronisation).
 *     Writes to a GEMM's weights from other streams must be ordered by the caller as usual.
 */
#ifndef WQL_H_
#define WQL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum wql_status {
  WQL_OK = 0,
  WQL_EINVAL = 1,        /* bad argument: shape, alignment, null pointer, group size */
  WQL_EUNSUPPORTED = 2,  /* valid request the library does not cover (e.g. K too large) */
  WQL_ECUDA = 3,         /* CUDA runtime/driver error at launch */
  WQL_ETIMEOUT = 4       /* a kernel's bounded on-chip wait expired (see wql_device_status) */
} wql_status;

/* Short constant description of a status code. */
const char* wql_status_string(int status);

/* Detail message of the last failing call on this host thread ("" if none). */
const char* wql_last_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
int wql_version(void);

/* Synchronises `stream`, then reports and clears the device-side error word of the current
 * device: WQL_ETIMEOUT if a kernel abandoned a bounded wait since the last check, WQL_ECUDA if
 * the synchronisation itself failed, WQL_OK otherwise. */
wql_status wql_device_status(void* stream);

/* Diagnostic of the failure path: launches one thread that waits on an on-chip barrier which
 * nothing completes.  Its bounded wait gives up after the same time limit as every kernel's
 * (about 2 s) and records the same device-side error, so the next wql_device_status() returns
 * WQL_ETIMEOUT (and clears it); the context stays usable.  Launches nothing else and touches no
 * caller memory.  Returns WQL_ECUDA if the launch fails. */
wql_status wql_diag_expire_wait(void* stream);

/* Phase trace of the W4A16 kernels, for a developer build compiled with -DWQL_PHASE_TRACE (a
 * library file of its own; the default build returns WQL_EUNSUPPORTED and does nothing).
 * Registers a device buffer buf of launches x ctas x 32 uint64 (caller-owned, zero-filled by the
 * caller): every later w4a16 launch whose output pointer y lies at ybase + l * ystride
 * (0 <= l < launches) writes, per CTA c < ctas, %globaltimer nanoseconds at its phase points into
 * buf[(l * ctas + c) * 32 + slot], and its SM id into slot 31.  Launches whose y lies elsewhere
 * are not recorded.  buf == NULL switches the trace off.  Stamps only: the kernels skip and
 * reorder nothing.  Call it between launches, not while one may be running. */
wql_status wql_trace_setup(uint64_t* buf, const void* ybase, uint64_t ystride, int launches, int ctas);

/* ----------------------------------------------------------------------------------------
 * awq_pack  [AWQ] section 2; [AUQ] sections 3.3 and 5.4.
 * Quantise fp32 weights w [K, N] to asymmetric int4, per group of G consecutive input
 * channels (k) and per output channel (n):
 *     s  = fp16((max_k w - min_k w) / 15)       (1.0 if that rounds to zero)
 *     z  = clamp(round(-min_k w / s), 0, 15)
 *     q  = clamp(round(w / s) + z, 0, 15)        round = half to even, fp32 arithmetic
 * so that w ~ (q - z) * s.  Outputs (all written in full):
 *     qweight [K, N/8] uint32: code of column n at bits 4*(n%8) of word n/8 of row k
 *     scales  [K/G, N] fp16
 *     qzeros  [K/G, N/8] uint32: zero points packed like qweight
 * Requires G in {32, 64, 128}, K % G == 0, N % 32 == 0, K >= 1.
 * ---------------------------------------------------------------------------------------- */
wql_status wql_awq_pack(const float* w, int K, int N, int group, uint32_t* qweight,
                        uint16_t* scales, uint32_t* qzeros, void* stream);

/* ----------------------------------------------------------------------------------------
 * w4a16_gemm  [AWQ] section 2, [TM] section 5.1.
 *     y[m, n] = sum_k x[m, k] * (q[k, n] - z[k/G, n]) * s[k/G, n]
 * x [M, K] fp16, packed weight as produced by wql_awq_pack, y [M, N] fp16 (written in full;
 * accumulation in fp32).  Decode-shaped calls (small M) stream the packed weight once with
 * tensor-core dot products; prefill-shaped calls use the tcgen05 tensor-core kernel.
 * Requires G in {32, 64, 128}, K % G == 0, N % 32 == 0, M >= 0.
 * ---------------------------------------------------------------------------------------- */
wql_status wql_w4a16_gemm(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                          const uint32_t* qzeros, int M, int K, int N, int group, uint16_t* y,
                          void* stream);

/* ----------------------------------------------------------------------------------------
 * w4a16_gemm_silu_mul  [FastLLM] section 2: the gate and up projections of an MLP as one GEMM,
 * with SiLU(gate) * up fused into its epilogue.  Reading: the packed weight (wql_awq_pack of a
 * [K, N] matrix) interleaves the projections by output channel -- channel 2j is gate j and
 * channel 2j + 1 is up j -- and
 *     y[m, j] = fp16(silu(g) * u),  g = fp16(gemm[m, 2j]),  u = fp16(gemm[m, 2j + 1]),
 *     silu(g) = g / (1 + exp(-g))   (fp32; IEEE division, expf)
 * i.e. exactly the unfused GEMM's fp16 outputs followed by the activation, without writing them.
 * x [M, K] fp16; y [M, N / 2] fp16.  Same kernels and requirements as wql_w4a16_gemm, and
 * N % 64 == 0.
 * ---------------------------------------------------------------------------------------- */
wql_status wql_w4a16_gemm_silu_mul(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                                   const uint32_t* qzeros, int M, int K, int N, int group, uint16_t* y,
                                   void* stream);

/* ----------------------------------------------------------------------------------------
 * w4a16_kernel_for: the kernel wql_w4a16_gemm runs for an M x K x N call with group size
 * `group` on the current device: 0 = the weight-streaming decode kernel, 1 = the tcgen05
 * tensor-core kernel.  Up to 16 tokens it is always 0 and from 33 on always 1; in between it
 * depends on N, K and the group size.  Host-only, never fails (the WQL_FORCE_KERNEL
 * benchmarking switch is not consulted).
 * ---------------------------------------------------------------------------------------- */
int wql_w4a16_kernel_for(int M, int K, int N, int group);

/* ----------------------------------------------------------------------------------------
 * qrmsnorm_quant_i8  [W8A8] QRMSNorm.forward + rms_norm_dynamic_quant / per_token_quant_int8.
 * Per row m of x [M, K] fp16, with gamma [K] fp16 (smoothing already folded in):
 *     ss   = sum_k x^2 in a fixed order: element k joins lane (k/8) % 256, lanes add in
 *            increasing k, then lanes fold pairwise (t, t+128), (t, t+64), ..., (t, t+1)
 *     r    = 1 / sqrt(ss / K + eps)
 *     y_k  = (x_k * r) * gamma_k            (fp32, one rounding per operation, kept in fp32)
 *     xs_m = max_k |y_k| / 127              (1.0 if the row is all zero)
 *     q_mk = clamp(round_half_even(y_k / xs_m), -128, 127)
 * Outputs q [M, K] int8 and xs [M] fp32, bit-exact with the definition above.
 * Requires K % 8 == 0, 8 <= K <= 16384.
 * ---------------------------------------------------------------------------------------- */
wql_status wql_qrmsnorm_quant_i8(const uint16_t* x, const uint16_t* gamma, float eps, int M,
                                 int K, int8_t* q, float* xs, void* stream);

/* ----------------------------------------------------------------------------------------
 * add_qrmsnorm_quant_i8  [W8A8] "inference kernels": rms_norm_dynamic_quant with its residual
 * fusion (add_rms_norm_quant_kernel).  The page names the fusion, not its arithmetic; reading:
 *     h[m, k] = fp16(float(x[m, k]) + float(residual[m, k]))   (one fp32 add, one rounding)
 * h is written to residual_out [M, K] fp16 (the new residual stream; residual_out may be the
 * residual buffer itself), and q [M, K] int8, xs [M] fp32 are QRMSNorm + per-token int8 of h,
 * exactly as wql_qrmsnorm_quant_i8 computes them for an input h.
 * Requires K % 8 == 0, 8 <= K <= 16384; every pointer 16-byte aligned (xs: 4-byte).
 * ---------------------------------------------------------------------------------------- */
wql_status wql_add_qrmsnorm_quant_i8(const uint16_t* x, const uint16_t* residual,
                                     const uint16_t* gamma, float eps, int M, int K,
                                     uint16_t* residual_out, int8_t* q, float* xs, void* stream);

/* ----------------------------------------------------------------------------------------
 * per_token_quant_i8 / per_token_quant_fp8  [W8A8] per_token_quant_int8, the quantiser
 * QLinear.forward applies when its input is a plain tensor rather than QRMSNorm's output.
 * Per row m of x [M, K] fp16, with x_k the fp16 value widened to fp32:
 *     xs_m = max_k |x_k| / Q_MAX    (Q_MAX = 127 for int8, 448 for e4m3; 1.0 if the row is zero)
 *     q_mk = clamp(round_half_even(x_k / xs_m), -128, 127)     (int8)
 *     q_mk = e4m3(x_k / xs_m)       (fp8: the e4m3 value nearest the fp32 quotient, ties to even)
 * Outputs q [M, K] (int8, or e4m3 bytes) and xs [M] fp32, bit-exact with the definition above;
 * (q, xs) feed wql_w8a8_gemm / wql_w8a8_gemm_fp8 as QRMSNorm's outputs do.
 * Requires K % 8 == 0, 8 <= K <= 16384 (WQL_EUNSUPPORTED above); x and q 16-byte aligned, xs
 * 4-byte aligned.
 * ---------------------------------------------------------------------------------------- */
wql_status wql_per_token_quant_i8(const uint16_t* x, int M, int K, int8_t* q, float* xs, void* stream);
wql_status wql_per_token_quant_fp8(const uint16_t* x, int M, int K, uint8_t* q, float* xs, void* stream);

/* ----------------------------------------------------------------------------------------
 * w8a8_gemm  [W8A8] QLinear.forward / matmul_kernel_dynamic_quant.
 *     acc[m, n] = sum_k q[m, k] * qw[n, k]                 (exact int32)
 *     y[m, n]   = fp16((float(acc[m, n]) * xs[m]) * ws[n])  (fp32, left to right)
 * q [M, K] int8 with per-token scales xs [M] fp32; qw [N, K] int8 (input dimension
 * contiguous, as a torch Linear weight) with per-channel scales ws [N] fp32.
 * y [M, N] fp16 is written in full; acc_out [M, N] int32 is written too when non-NULL.
 * The int32 result is exact for every input (|acc| < 2^31 holds for K <= 131072).
 * workspace: device scratch of at least wql_w8a8_workspace_bytes(M, K, N) bytes (M * K * 2 +
 * 16384 for M >= 17: an fp16 copy of q and the largest row L1 norms of q; 0 below), used only
 * during the call (may be NULL when that size is 0).
 * Requires K % 16 == 0, N % 32 == 0, M >= 0, K <= 131072.
 * ---------------------------------------------------------------------------------------- */
size_t wql_w8a8_workspace_bytes(int M, int K, int N);
wql_status wql_w8a8_gemm(const int8_t* q, const float* xs, const int8_t* qw, const float* ws,
                         int M, int K, int N, uint16_t* y, int32_t* acc_out, void* workspace,
                         size_t workspace_bytes, void* stream);

/* ----------------------------------------------------------------------------------------
 * w8a8_gemm_fused  [W8A8] "inference kernels": the _linear_add variant of
 * matmul_kernel_dynamic_quant with its optional bias and residual.  The page names the
 * fusion, not its arithmetic; reading:
 *     y[m, n] = fp16(((float(acc[m, n]) * xs[m]) * ws[n] + float(bias[n])) + float(residual[m, n]))
 * in fp32, left to right, one rounding to fp16.  bias [N] fp16 and residual [M, N] fp16 are
 * each optional (NULL leaves the term out); residual may be y itself (in place).  Everything
 * else, including acc_out and the workspace, is as for wql_w8a8_gemm.
 * ---------------------------------------------------------------------------------------- */
wql_status wql_w8a8_gemm_fused(const int8_t* q, const float* xs, const int8_t* qw, const float* ws,
                               const uint16_t* bias, const uint16_t* residual, int M, int K, int N,
                               uint16_t* y, int32_t* acc_out, void* workspace,
                               size_t workspace_bytes, void* stream);

/* ----------------------------------------------------------------------------------------
 * w8a8_gemm_noalloc -- the same operation as wql_w8a8_gemm (same kernels, same results) for
 * callers that cannot allocate device memory at call time: an engine that has already handed
 * its whole memory budget to its own pool, a plugin whose host framework owns every allocation,
 * or a latency-critical loop that must not pay for the allocator's synchronisation.  The source
 * pages have no counterpart to this entry point; it exists for such callers only.
 * Instead of a caller workspace it uses a scratch array built into the library:
 *   - 32 MiB + 64 KiB, so M * K * 2 + 16384 <= 33619968 (e.g. M = K = 4096); larger calls return
 *     WQL_EUNSUPPORTED with a message in wql_last_error() and launch nothing;
 *   - one array per GPU that loads the library, held until the process exits;
 *   - the first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current) and keeps it; make that first call before any stream capture.
 *     cudaDeviceReset invalidates the kept address: no call may follow a reset of that device
 *     in the same process;
 *   - every call on a device shares the one array.  Calls that may overlap on the GPU (other
 *     streams, other threads) race on it and must be serialised by the caller.  Nothing in it
 *     needs to start at zero: each call overwrites every byte it later reads.
 * The library allocates and frees nothing in this call.
 * ---------------------------------------------------------------------------------------- */
wql_status wql_w8a8_gemm_noalloc(const int8_t* q, const float* xs, const int8_t* qw,
                                 const float* ws, int M, int K, int N, uint16_t* y,
                                 int32_t* acc_out, void* stream);

/* ----------------------------------------------------------------------------------------
 * Offline preparation for W8A8 ([W8A8] "weight smoothing" and QLinear.from_float).
 *
 * wql_act_absmax: calibration statistic a_j = max_m |RMSNorm_gamma(x)[m, j]| over x [M, K]
 *   (same fp32 RMSNorm as wql_qrmsnorm_quant_i8, original gamma).  absmax [K] fp32 is
 *   overwritten.  Requires K % 8 == 0, 8 <= K <= 16384.
 * wql_smooth: smooth_ln_fcs with alpha = 0.5 for one norm feeding one linear w [K, N] fp32:
 *     w_j = max_n |w[j, n]|;  s_j = sqrt(a_j / w_j)  (1 where a_j or w_j is 0)
 *     gamma_out_j = fp16(gamma_j / s_j);  w_out[j, n] = w[j, n] * s_j
 *   Outputs s [K] fp32, gamma_out [K] fp16, w_out [K, N] fp32 (may alias w).
 * wql_per_channel_quant_i8: ws_n = max_k |w[k, n]| / 127 (1.0 for a zero column);
 *     qw[n, k] = clamp(round_half_even(w[k, n] / ws_n), -127, 127)
 *   w [K, N] fp32 -> qw [N, K] int8 (transposed), ws [N] fp32.
 * Requires K % 16 == 0, N % 32 == 0.
 * ---------------------------------------------------------------------------------------- */
wql_status wql_act_absmax(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K,
                          float* absmax, void* stream);
wql_status wql_smooth(const float* absmax, const uint16_t* gamma, const float* w, int K, int N,
                      float* s, uint16_t* gamma_out, float* w_out, void* stream);
wql_status wql_per_channel_quant_i8(const float* w, int K, int N, int8_t* qw, float* ws,
                                    void* stream);

/* ========================================================================================
 * FP8 variant of W8A8 ([W8A8]: quant_dtype "fp8", the short name of float8_e4m3fn).
 * Codes are float8 e4m3 bytes (1 sign, 4 exponent bits with bias 7, 3 fraction bits, no
 * infinity, largest value 448), passed as uint8_t.  Q_MAX = 448 (torch.finfo of the type)
 * replaces 127, and the page casts instead of rounding to an integer.  Reading of the cast:
 * nearest e4m3 value, ties to even, magnitudes beyond 448 saturated to 448.
 * ======================================================================================== */

/* ----------------------------------------------------------------------------------------
 * qrmsnorm_quant_fp8: wql_qrmsnorm_quant_i8 with fp8 codes.  y is the same fp32 RMSNorm;
 *     xs[m]   = max_k |y[m, k]| / 448   (1.0 for an all-zero row)
 *     q[m, k] = e4m3(y[m, k] / xs[m])   (the quotient correctly rounded in fp32 first)
 * add_qrmsnorm_quant_fp8: the residual fusion, exactly as wql_add_qrmsnorm_quant_i8 (h =
 * fp16(x + residual) goes to residual_out, which may be residual itself) with fp8 codes.
 * Requires K % 8 == 0, 8 <= K <= 16384; every pointer 16-byte aligned (xs: 4-byte).
 * ---------------------------------------------------------------------------------------- */
wql_status wql_qrmsnorm_quant_fp8(const uint16_t* x, const uint16_t* gamma, float eps, int M, int K,
                                  uint8_t* q, float* xs, void* stream);
wql_status wql_add_qrmsnorm_quant_fp8(const uint16_t* x, const uint16_t* residual,
                                      const uint16_t* gamma, float eps, int M, int K,
                                      uint16_t* residual_out, uint8_t* q, float* xs, void* stream);

/* ----------------------------------------------------------------------------------------
 * per_channel_quant_fp8: ws_n = max_k |w[k, n]| / 448 (1.0 for a zero column);
 *     qw[n, k] = e4m3(w[k, n] / ws_n)
 *   w [K, N] fp32 -> qw [N, K] e4m3 (transposed), ws [N] fp32.  Requires K % 16 == 0, N % 32 == 0.
 * ---------------------------------------------------------------------------------------- */
wql_status wql_per_channel_quant_fp8(const float* w, int K, int N, uint8_t* qw, float* ws,
                                     void* stream);

/* ----------------------------------------------------------------------------------------
 * w8a8_gemm_fp8  [W8A8] matmul_kernel_dynamic_quant with fp8 inputs (fp32 accumulator) and
 * the optional terms of its _linear_add variant:
 *     acc[m, n] = sum_k e4m3(q[m, k]) * e4m3(qw[n, k])       (fp32 accumulation)
 *     y[m, n]   = fp16(((acc[m, n] * xs[m]) * ws[n] + float(bias[n])) + float(residual[m, n]))
 * q [M, K], qw [N, K] e4m3; xs [M], ws [N] fp32; bias [N] and residual [M, N] fp16, each
 * optional (NULL leaves the term out; residual may be y itself).  y [M, N] fp16 is written in
 * full, and acc_out [M, N] fp32 too when non-NULL.  The order of the fp32 additions is the
 * kernel's own (tensor-core sums, then a fixed-order split-K reduction), so acc differs from
 * the exact sum by at most K * 2^-23 * sum_k |product| -- an fp32 rounding per addition.
 * No workspace.  Requires K % 16 == 0, N % 32 == 0, M >= 0.
 * ---------------------------------------------------------------------------------------- */
wql_status wql_w8a8_gemm_fp8(const uint8_t* q, const float* xs, const uint8_t* qw, const float* ws,
                             const uint16_t* bias, const uint16_t* residual, int M, int K, int N,
                             uint16_t* y, float* acc_out, void* stream);

/* ========================================================================================
 * KV cache int8 in groups of 128 ([FastLLM] section 5.2: the K and V cache stored as int8 with
 * group size 128, dequantised when read).  The page fixes the width and the group size only.
 * Reading: a group is 128 consecutive channels of one row (one token's K or V vector),
 * symmetric like [W8A8]'s per-token int8:
 *     scales[r, g] = max_{k in group g} |kv[r, k]| / 127      (fp32; 1.0 for an all-zero group)
 *     q[r, k]      = clamp(round_half_even(kv[r, k] / scales[r, k / 128]), -128, 127)
 * and the cache entry read back is out[r, k] = fp16(float(q[r, k]) * scales[r, k / 128]).
 * kv and out are [rows, D] fp16, q is [rows, D] int8, scales [rows, D / 128] fp32, all row-major
 * and contiguous (rows may count tokens x layers; a row is any run of D channels).
 * Requires D % 128 == 0, rows >= 0 (0 is a no-op); pointers 16-byte aligned (scales: 4-byte).
 * ======================================================================================== */
wql_status wql_kv_quant_i8(const uint16_t* kv, int64_t rows, int D, int8_t* q, float* scales,
                           void* stream);
wql_status wql_kv_dequant_i8(const int8_t* q, const float* scales, int64_t rows, int D,
                             uint16_t* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* WQL_H_ */
