/*
 * wql_oracle.c -- plain, slow CPU reference for the weight-quantized linear layers.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path may include, link or call this
 * file; only the test-suite, the smoke check and the benchmark's CPU-baseline leg do.  It
 * shares no code, header, table or helper with the CUDA sources.
 *
 * Built with `gcc -O2 -ffp-contract=off -fopenmp` so that every float expression below is
 * evaluated as written: one IEEE-754 binary32 rounding per operation, no fused multiply-add.
 *
 * Sources (page titles of the public write-ups this restates):
 *   [AWQ]  "LMDeploy ... INT4 quantisation" tutorial, section 2 (asymmetric per-group min/max
 *          scale and zero point; group sizes 32/64/128; `--w-bits 4 --w-group-size 128`).
 *   [AUQ]  "AUQ dual-process framework" article, section 3.3 (AWQ dequant uses a per-group
 *          scale and zero point) and section 5.4 (checkpoint tensors qweight/scales/zeros,
 *          qweight dim 0 divisible by 128, i.e. dim 0 is the grouped input dimension).
 *   [W8A8] "LMDeploy W8A8 quantisation guide", sections "weight smoothing" (smooth_ln_fcs,
 *          alpha = 0.5), "QRMSNorm / QLinear" (per-token dynamic quant, per-channel weight
 *          quant with fp32 scales) and "inference kernels" (per_token_quant_int8: scale =
 *          absmax / Q_MAX with Q_MAX = 127 for int8, values rounded to integers;
 *          matmul_kernel_dynamic_quant: int32 accumulator, c = c * rms_scale * linear_scale),
 *          and its fp8 variant (quant_dtype fp8 = float8_e4m3fn, Q_MAX from torch.finfo, values
 *          cast instead of rounded to integers, fp32 accumulator).
 *   [FastLLM] "FastLLM architecture" article, section 2 (fused gate/up GEMM followed by SiLU * up)
 *          and section 5.2 (KV cache quantised to int8 in groups of 128, dequantised when read).
 *
 * Readings taken where the pages are silent (each one is listed in the design notes):
 *   - zero point is an integer z in [0,15] stored 8 per uint32 like the codes; w ~ (q - z) * s;
 *   - column n of a packed word sits at bits 4*(n % 8) of word n / 8;
 *   - the scale is rounded to fp16 before z and q are derived from it; a zero fp16 scale is
 *     replaced by 1.0;
 *   - rounding is round-half-to-even everywhere;
 *   - RMSNorm: r = 1 / sqrt(mean(x^2) + eps), y = (x * r) * gamma, kept in fp32 (fused, never
 *     stored as fp16 before quantisation); the sum of squares follows the fixed order of
 *     wql_oracle_sumsq below so that int8 codes can be compared bit for bit;
 *   - an all-zero row gets scale 1.0 (all codes 0); weights are clamped to [-127, 127];
 *   - smoothing statistics are the per-channel absmax of RMSNorm_gamma(X) on the same batch;
 *   - the fp8 cast rounds to the nearest e4m3 value (ties to even) and saturates at +-448.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------------------
 * IEEE-754 binary16 <-> binary32, written from the format's definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits; subnormals scale 2^-24).
 * ------------------------------------------------------------------------------------- */
float wql_oracle_half_to_float(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 31;
  const int f = h & 1023;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25);
  }
  return (float)(sign ? -v : v);
}

uint16_t wql_oracle_float_to_half(float x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
  double a = fabs((double)x);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u); /* rounds past the largest finite */
  if (a < ldexp(1.0, -14)) {
    /* subnormal (or zero): units of 2^-24, ties to even; 1024 units is the smallest normal */
    double units = nearbyint(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)units);
  }
  int e2;
  frexp(a, &e2);            /* a = m * 2^e2, m in [0.5, 1) => a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;           /* unbiased exponent */
  double sig = nearbyint(ldexp(a, 10 - E)); /* in [1024, 2048], ties to even */
  if (sig >= 2048.0) { sig = 1024.0; E += 1; }
  if (E + 15 >= 31) return (uint16_t)(sign | 0x7c00u);
  return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(sig - 1024.0));
}

void wql_oracle_half_to_float_n(const uint16_t* h, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = wql_oracle_half_to_float(h[i]);
}
void wql_oracle_float_to_half_n(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = wql_oracle_float_to_half(x[i]);
}

int wql_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* round half to even, then clamp to [lo, hi], without ever converting an out-of-range float */
static int clamp_rint(float v, float lo, float hi) {
  float r = nearbyintf(v);
  if (!(r >= lo)) r = lo; /* also catches NaN */
  if (r > hi) r = hi;
  return (int)r;
}

/* ---------------------------------------------------------------------------------------
 * [AWQ] section 2, [AUQ] sections 3.3 / 5.4: asymmetric per-group int4 quantisation.
 * W is [K, N] row-major fp32 (K = input features, grouped in runs of `group` along K).
 * Outputs: qweight [K, N/8] u32, scales [K/group, N] fp16 bits, qzeros [K/group, N/8] u32.
 * ------------------------------------------------------------------------------------- */
void wql_oracle_awq_quantize(const float* W, int K, int N, int group,
                             uint32_t* qweight, uint16_t* scales, uint32_t* qzeros) {
  const int ngroups = K / group;
  memset(qweight, 0, sizeof(uint32_t) * (size_t)K * (N / 8));
  memset(qzeros, 0, sizeof(uint32_t) * (size_t)ngroups * (N / 8));
#pragma omp parallel for schedule(static)
  for (int g = 0; g < ngroups; ++g) {
    for (int n = 0; n < N; ++n) {
      /* step 1: the group's own minimum and maximum (zero is not forced into the range) */
      float mn = W[(size_t)(g * group) * N + n], mx = mn;
      for (int k = g * group + 1; k < (g + 1) * group; ++k) {
        float w = W[(size_t)k * N + n];
        if (w < mn) mn = w;
        if (w > mx) mx = w;
      }
      /* step 2: scale spreads the range over the 15 steps of a 4-bit code, stored as fp16 */
      float s32 = (mx - mn) / 15.0f;
      uint16_t s16 = wql_oracle_float_to_half(s32);
      if ((s16 & 0x7fffu) == 0) s16 = 0x3c00u; /* degenerate (constant) group: scale 1.0 */
      float s = wql_oracle_half_to_float(s16);
      /* step 3: integer zero point puts the minimum at code 0 */
      int z = clamp_rint(-mn / s, 0.0f, 15.0f);
      scales[(size_t)g * N + n] = s16;
      qzeros[(size_t)g * (N / 8) + n / 8] |= (uint32_t)z << (4 * (n % 8));
      /* step 4: codes q = round(w / s) + z, clamped to the 4-bit range */
      for (int k = g * group; k < (g + 1) * group; ++k) {
        float w = W[(size_t)k * N + n];
        float t = nearbyintf(w / s) + (float)z;
        int q = clamp_rint(t, 0.0f, 15.0f);
        qweight[(size_t)k * (N / 8) + n / 8] |= (uint32_t)q << (4 * (n % 8));
      }
    }
  }
}

/* Unpack codes and zero points into one byte per element: q [K, N], z [K/group, N]. */
void wql_oracle_awq_unpack(const uint32_t* qweight, const uint32_t* qzeros, int K, int N,
                           int group, uint8_t* q, uint8_t* z) {
  for (int k = 0; k < K; ++k)
    for (int n = 0; n < N; ++n)
      q[(size_t)k * N + n] = (qweight[(size_t)k * (N / 8) + n / 8] >> (4 * (n % 8))) & 15u;
  for (int g = 0; g < K / group; ++g)
    for (int n = 0; n < N; ++n)
      z[(size_t)g * N + n] = (qzeros[(size_t)g * (N / 8) + n / 8] >> (4 * (n % 8))) & 15u;
}

/* Dequantise one row k of the packed weight: w[n] = (q - z) * s, in fp32 (exact: a 5-bit
 * integer times an fp16 value needs at most 16 significant bits). */
static void dequant_row(const uint32_t* qweight, const uint16_t* scales, const uint32_t* qzeros,
                        int N, int group, int k, float* out) {
  const int g = k / group;
  for (int n = 0; n < N; ++n) {
    int q = (qweight[(size_t)k * (N / 8) + n / 8] >> (4 * (n % 8))) & 15;
    int z = (qzeros[(size_t)g * (N / 8) + n / 8] >> (4 * (n % 8))) & 15;
    float s = wql_oracle_half_to_float(scales[(size_t)g * N + n]);
    out[n] = (float)(q - z) * s;
  }
}

void wql_oracle_awq_dequant(const uint32_t* qweight, const uint16_t* scales,
                            const uint32_t* qzeros, int K, int N, int group, float* w) {
  for (int k = 0; k < K; ++k) dequant_row(qweight, scales, qzeros, N, group, k, w + (size_t)k * N);
}

/* ---------------------------------------------------------------------------------------
 * W4A16 linear: Y[m, n] = sum_k X[m, k] * (q[k, n] - z[k/G, n]) * s[k/G, n].
 * Weights dequantised to fp32, products and sums in fp64, accumulated in increasing k.
 * `rows` (length nrows) selects which rows of X/Y to compute; Y is [nrows, N] fp64.
 * ------------------------------------------------------------------------------------- */
void wql_oracle_w4a16_linear(const uint16_t* X, const uint32_t* qweight, const uint16_t* scales,
                             const uint32_t* qzeros, int K, int N, int group,
                             const int64_t* rows, int nrows, double* Y) {
  memset(Y, 0, sizeof(double) * (size_t)nrows * N);
  float* wrow = (float*)malloc(sizeof(float) * (size_t)N);
  double* xcol = (double*)malloc(sizeof(double) * (size_t)nrows);
  for (int k = 0; k < K; ++k) {
    dequant_row(qweight, scales, qzeros, N, group, k, wrow);
    for (int i = 0; i < nrows; ++i) xcol[i] = (double)wql_oracle_half_to_float(X[(size_t)rows[i] * K + k]);
#pragma omp parallel for schedule(static)
    for (int i = 0; i < nrows; ++i) {
      const double xv = xcol[i];
      double* y = Y + (size_t)i * N;
      for (int n = 0; n < N; ++n) y[n] += xv * (double)wrow[n];
    }
  }
  free(wrow);
  free(xcol);
}

/* ---------------------------------------------------------------------------------------
 * [W8A8] QRMSNorm: the sum of squares of one row, in a fixed order.
 * Element k belongs to lane (k / 8) mod 256; each lane adds its elements in increasing k;
 * the 256 lane sums are then folded pairwise (t, t + 128), (t, t + 64), ..., (t, t + 1).
 * Each x^2 is exact in fp32 (an fp16 significand has 11 bits); every addition rounds once.
 * ------------------------------------------------------------------------------------- */
float wql_oracle_sumsq(const uint16_t* x, int K) {
  float lane[256];
  for (int t = 0; t < 256; ++t) lane[t] = 0.0f;
  for (int k = 0; k < K; ++k) {
    float v = wql_oracle_half_to_float(x[k]);
    int t = (k / 8) % 256;
    lane[t] = lane[t] + v * v;
  }
  for (int stride = 128; stride >= 1; stride /= 2)
    for (int t = 0; t < stride; ++t) lane[t] = lane[t] + lane[t + stride];
  return lane[0];
}

/* r = 1 / sqrt(mean(x^2) + eps), one rounding per operation. */
static float rms_factor(const uint16_t* x, int K, float eps) {
  float ss = wql_oracle_sumsq(x, K);
  float mean = ss / (float)K;
  float d = sqrtf(mean + eps);
  return 1.0f / d;
}

/* y = RMSNorm_gamma(x) in fp32: y_k = (x_k * r) * gamma_k; out is [M, K] fp32. */
void wql_oracle_rmsnorm(const uint16_t* X, const uint16_t* gamma, float eps, int M, int K,
                        float* out) {
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m) {
    const uint16_t* x = X + (size_t)m * K;
    float r = rms_factor(x, K, eps);
    for (int k = 0; k < K; ++k) {
      float t = wql_oracle_half_to_float(x[k]) * r;
      out[(size_t)m * K + k] = t * wql_oracle_half_to_float(gamma[k]);
    }
  }
}

/* [W8A8] QRMSNorm fused with per-token dynamic int8 quantisation:
 * xs_m = max_k |y_mk| / 127 (1.0 for an all-zero row); q_mk = clamp(rint(y_mk / xs_m), -128, 127). */
void wql_oracle_qrmsnorm_quant_i8(const uint16_t* X, const uint16_t* gamma, float eps, int M,
                                  int K, int8_t* q, float* xs) {
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m) {
    const uint16_t* x = X + (size_t)m * K;
    float r = rms_factor(x, K, eps);
    float* y = (float*)malloc(sizeof(float) * (size_t)K);
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
      float t = wql_oracle_half_to_float(x[k]) * r;
      y[k] = t * wql_oracle_half_to_float(gamma[k]);
      float a = fabsf(y[k]);
      if (a > amax) amax = a;
    }
    float scale = amax / 127.0f;
    if (amax == 0.0f) scale = 1.0f;
    xs[m] = scale;
    for (int k = 0; k < K; ++k) q[(size_t)m * K + k] = (int8_t)clamp_rint(y[k] / scale, -128.0f, 127.0f);
    free(y);
  }
}

/* [W8A8] per_token_quant_int8, the quantiser QLinear.forward applies to an input that does not come
 * from QRMSNorm: the same per-token rule on the activations themselves,
 * xs_m = max_k |x_mk| / 127 (1.0 for an all-zero row); q_mk = clamp(rint(x_mk / xs_m), -128, 127),
 * with x_mk the fp16 value widened to fp32 and one rounding per operation. */
void wql_oracle_per_token_quant_i8(const uint16_t* X, int M, int K, int8_t* q, float* xs) {
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m) {
    const uint16_t* x = X + (size_t)m * K;
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
      float a = fabsf(wql_oracle_half_to_float(x[k]));
      if (a > amax) amax = a;
    }
    float scale = amax / 127.0f;
    if (amax == 0.0f) scale = 1.0f;
    xs[m] = scale;
    for (int k = 0; k < K; ++k)
      q[(size_t)m * K + k] = (int8_t)clamp_rint(wql_oracle_half_to_float(x[k]) / scale, -128.0f, 127.0f);
  }
}

/* [W8A8] calibration statistic used by smoothing: a_j = max_m |RMSNorm_gamma(X)_mj|. */
/* [W8A8] "inference kernels": rms_norm_dynamic_quant with its residual fusion
 * (add_rms_norm_quant_kernel).  Reading (the page names the fusion, not its arithmetic):
 * h = fp16(float(x) + float(r)) -- one fp32 addition of the two fp16 values, rounded to fp16 --
 * is the new residual stream H, and the row that is normalised and quantised, exactly as
 * wql_oracle_qrmsnorm_quant_i8 does for an unfused input. */
void wql_oracle_add_qrmsnorm_quant_i8(const uint16_t* X, const uint16_t* R, const uint16_t* gamma,
                                     float eps, int M, int K, uint16_t* H, int8_t* q, float* xs) {
  for (int64_t i = 0; i < (int64_t)M * K; ++i) {
    float sum = wql_oracle_half_to_float(X[i]) + wql_oracle_half_to_float(R[i]);
    H[i] = wql_oracle_float_to_half(sum);
  }
  wql_oracle_qrmsnorm_quant_i8(H, gamma, eps, M, K, q, xs);
}

void wql_oracle_act_absmax(const uint16_t* X, const uint16_t* gamma, float eps, int M, int K,
                           float* absmax) {
  float* y = (float*)malloc(sizeof(float) * (size_t)M * K);
  wql_oracle_rmsnorm(X, gamma, eps, M, K, y);
  for (int k = 0; k < K; ++k) absmax[k] = 0.0f;
  for (int m = 0; m < M; ++m)
    for (int k = 0; k < K; ++k) {
      float a = fabsf(y[(size_t)m * K + k]);
      if (a > absmax[k]) absmax[k] = a;
    }
  free(y);
}

/* [W8A8] smooth_ln_fcs with alpha = 0.5 for one RMSNorm feeding one linear layer W [K, N]:
 *   w_j = max_n |W[j, n]|,  s_j = sqrt(a_j / w_j)  (= a_j^0.5 / w_j^0.5; 1 where a_j or w_j is 0),
 *   gamma'_j = fp16(gamma_j / s_j),  W'[j, n] = W[j, n] * s_j. */
void wql_oracle_smooth(const float* absmax, const uint16_t* gamma, const float* W, int K, int N,
                       float* s_out, uint16_t* gamma_out, float* W_out) {
#pragma omp parallel for schedule(static)
  for (int j = 0; j < K; ++j) {
    float wmax = 0.0f;
    for (int n = 0; n < N; ++n) {
      float a = fabsf(W[(size_t)j * N + n]);
      if (a > wmax) wmax = a;
    }
    float s = 1.0f;
    if (absmax[j] > 0.0f && wmax > 0.0f) s = sqrtf(absmax[j] / wmax);
    s_out[j] = s;
    gamma_out[j] = wql_oracle_float_to_half(wql_oracle_half_to_float(gamma[j]) / s);
    for (int n = 0; n < N; ++n) W_out[(size_t)j * N + n] = W[(size_t)j * N + n] * s;
  }
}

/* [W8A8] per_channel_quant: one fp32 scale per output channel n,
 * ws_n = max_k |W[k, n]| / 127 (1.0 for an all-zero column); qW[n, k] = clamp(rint(W[k, n] / ws_n), -127, 127).
 * Output qW is [N, K] (input dimension contiguous, as a torch Linear weight). */
void wql_oracle_per_channel_quant_i8(const float* W, int K, int N, int8_t* qW, float* ws) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
      float a = fabsf(W[(size_t)k * N + n]);
      if (a > amax) amax = a;
    }
    float scale = amax / 127.0f;
    if (amax == 0.0f) scale = 1.0f;
    ws[n] = scale;
    for (int k = 0; k < K; ++k)
      qW[(size_t)n * K + k] = (int8_t)clamp_rint(W[(size_t)k * N + n] / scale, -127.0f, 127.0f);
  }
}

/* [W8A8] integer GEMM: acc[i, n] = sum_k q[rows[i], k] * qW[n, k], exact in int64.
 * Returns 0 if every result fits int32, 1 otherwise (then acc holds the low 32 bits). */
int wql_oracle_w8a8_acc(const int8_t* q, const int8_t* qW, int K, int N, const int64_t* rows,
                        int nrows, int32_t* acc) {
  int overflow = 0;
#pragma omp parallel for schedule(static) reduction(| : overflow)
  for (int i = 0; i < nrows; ++i) {
    const int8_t* a = q + (size_t)rows[i] * K;
    for (int n = 0; n < N; ++n) {
      const int8_t* b = qW + (size_t)n * K;
      int64_t s = 0;
      for (int k = 0; k < K; ++k) s += (int64_t)a[k] * (int64_t)b[k];
      if (s > INT32_MAX || s < INT32_MIN) overflow = 1;
      acc[(size_t)i * N + n] = (int32_t)s;
    }
  }
  return overflow;
}

/* [W8A8] dequantising epilogue, c = c * rms_scale * linear_scale, in fp32 left to right,
 * then rounded to fp16: y = fp16((float(acc) * xs_m) * ws_n). xs holds the selected rows. */
void wql_oracle_w8a8_epilogue(const int32_t* acc, const float* xs, const float* ws, int nrows,
                              int N, uint16_t* y) {
  for (int i = 0; i < nrows; ++i)
    for (int n = 0; n < N; ++n) {
      float c = (float)acc[(size_t)i * N + n];
      float t = c * xs[i];
      y[(size_t)i * N + n] = wql_oracle_float_to_half(t * ws[n]);
    }
}

/* [W8A8] "inference kernels": matmul_kernel_dynamic_quant's _linear_add variant, with the
 * optional bias and residual the page names.  Reading (the page names the fusion, not its
 * arithmetic): the plain epilogue's fp32 value, then + bias[n], then + residual[i, n] (each an
 * fp16 value widened to fp32), left to right, one rounding to fp16 at the end.  A NULL bias or
 * residual leaves its term out altogether (adding 0.0 would turn a -0.0 result into +0.0). */
void wql_oracle_w8a8_epilogue_fused(const int32_t* acc, const float* xs, const float* ws,
                                    const uint16_t* bias, const uint16_t* residual, int nrows, int N,
                                    uint16_t* y) {
  for (int i = 0; i < nrows; ++i)
    for (int n = 0; n < N; ++n) {
      float c = (float)acc[(size_t)i * N + n];
      float t = c * xs[i];
      float u = t * ws[n];
      if (bias) u = u + wql_oracle_half_to_float(bias[n]);
      if (residual) u = u + wql_oracle_half_to_float(residual[(size_t)i * N + n]);
      y[(size_t)i * N + n] = wql_oracle_float_to_half(u);
    }
}

/* Same epilogue in fp64 without the final rounding, for tolerance checks. */
void wql_oracle_w8a8_epilogue_f64(const int32_t* acc, const float* xs, const float* ws,
                                  int nrows, int N, double* y) {
  for (int i = 0; i < nrows; ++i)
    for (int n = 0; n < N; ++n)
      y[(size_t)i * N + n] = (double)acc[(size_t)i * N + n] * (double)xs[i] * (double)ws[n];
}

/* ---------------------------------------------------------------------------------------
 * [W8A8] FP8 variant: quant_dtype "fp8", the short name of float8_e4m3fn.  The format, from
 * its definition: 1 sign bit, 4 exponent bits with bias 7, 3 fraction bits; exponent field 0
 * holds the subnormals, in units of 2^-9; there is no infinity and only S.1111.111 is NaN, so
 * the largest finite magnitude is 1.75 * 2^8 = 448 -- the Q_MAX that torch.finfo gives.
 * ------------------------------------------------------------------------------------- */
float wql_oracle_e4m3_to_float(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, f = b & 7;
  double v;
  if (e == 15 && f == 7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)f, -9);
  } else {
    v = ldexp((double)(8 + f), e - 10); /* (1 + f/8) * 2^(e-7) */
  }
  return (float)(sign ? -v : v);
}

/* Reading of the page's "FP8 is cast directly instead of being rounded to an integer": the
 * value goes to the nearest e4m3 number, ties to even (the default rounding of a float cast),
 * and a magnitude of 448 or more saturates to 448 (the codes come from x / (absmax / 448), which
 * can exceed 448 only by the rounding of that quotient).  NaN stays NaN. */
uint8_t wql_oracle_float_to_e4m3(float x) {
  const uint8_t sign = signbit(x) ? 0x80u : 0u;
  if (isnan(x)) return (uint8_t)(sign | 0x7fu);
  const double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7eu);
  if (a < ldexp(1.0, -6)) {
    /* subnormal (or zero): units of 2^-9, ties to even; 8 units is the smallest normal, 0x08 */
    const double units = nearbyint(ldexp(a, 9));
    return (uint8_t)(sign | (uint8_t)units);
  }
  int e2;
  frexp(a, &e2); /* a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;
  double sig = nearbyint(ldexp(a, 3 - E)); /* in [8, 16], ties to even */
  if (sig >= 16.0) {
    sig = 8.0;
    E += 1;
  }
  /* a < 448 keeps E <= 8 and sig <= 14 at E = 8, so the code is finite */
  return (uint8_t)(sign | (uint8_t)((E + 7) << 3) | (uint8_t)(sig - 8.0));
}

void wql_oracle_e4m3_to_float_n(const uint8_t* b, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = wql_oracle_e4m3_to_float(b[i]);
}
void wql_oracle_float_to_e4m3_n(const float* x, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = wql_oracle_float_to_e4m3(x[i]);
}

/* [W8A8] QRMSNorm with per-token dynamic fp8 quantisation: the same normalised row y as the int8
 * variant; xs_m = max_k |y_mk| / 448 (1.0 for an all-zero row); q_mk = e4m3(y_mk / xs_m). */
void wql_oracle_qrmsnorm_quant_fp8(const uint16_t* X, const uint16_t* gamma, float eps, int M,
                                   int K, uint8_t* q, float* xs) {
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m) {
    const uint16_t* x = X + (size_t)m * K;
    float r = rms_factor(x, K, eps);
    float* y = (float*)malloc(sizeof(float) * (size_t)K);
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
      float t = wql_oracle_half_to_float(x[k]) * r;
      y[k] = t * wql_oracle_half_to_float(gamma[k]);
      float a = fabsf(y[k]);
      if (a > amax) amax = a;
    }
    float scale = amax / 448.0f;
    if (amax == 0.0f) scale = 1.0f;
    xs[m] = scale;
    for (int k = 0; k < K; ++k) q[(size_t)m * K + k] = wql_oracle_float_to_e4m3(y[k] / scale);
    free(y);
  }
}

/* The fp8 twin of per_token_quant_int8: xs_m = max_k |x_mk| / 448 (1.0 for an all-zero row);
 * q_mk = e4m3(x_mk / xs_m), the e4m3 value nearest the fp32 quotient (ties to even). */
void wql_oracle_per_token_quant_fp8(const uint16_t* X, int M, int K, uint8_t* q, float* xs) {
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m) {
    const uint16_t* x = X + (size_t)m * K;
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
      float a = fabsf(wql_oracle_half_to_float(x[k]));
      if (a > amax) amax = a;
    }
    float scale = amax / 448.0f;
    if (amax == 0.0f) scale = 1.0f;
    xs[m] = scale;
    for (int k = 0; k < K; ++k) q[(size_t)m * K + k] = wql_oracle_float_to_e4m3(wql_oracle_half_to_float(x[k]) / scale);
  }
}

/* The residual fusion of the fp8 variant: h = fp16(float(x) + float(r)) as for int8, then the
 * fp8 QRMSNorm of h. */
void wql_oracle_add_qrmsnorm_quant_fp8(const uint16_t* X, const uint16_t* R, const uint16_t* gamma,
                                       float eps, int M, int K, uint16_t* H, uint8_t* q, float* xs) {
  for (int64_t i = 0; i < (int64_t)M * K; ++i) {
    float sum = wql_oracle_half_to_float(X[i]) + wql_oracle_half_to_float(R[i]);
    H[i] = wql_oracle_float_to_half(sum);
  }
  wql_oracle_qrmsnorm_quant_fp8(H, gamma, eps, M, K, q, xs);
}

/* [W8A8] per_channel_quant into fp8: ws_n = max_k |W[k, n]| / 448 (1.0 for an all-zero column),
 * qW[n, k] = e4m3(W[k, n] / ws_n), stored [N, K]. */
void wql_oracle_per_channel_quant_fp8(const float* W, int K, int N, uint8_t* qW, float* ws) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
      float a = fabsf(W[(size_t)k * N + n]);
      if (a > amax) amax = a;
    }
    float scale = amax / 448.0f;
    if (amax == 0.0f) scale = 1.0f;
    ws[n] = scale;
    for (int k = 0; k < K; ++k) qW[(size_t)n * K + k] = wql_oracle_float_to_e4m3(W[(size_t)k * N + n] / scale);
  }
}

/* [W8A8] fp8 GEMM: the page's kernel takes an fp32 accumulator when its inputs are floating point.
 * The reference is the exact sum acc[i, n] = sum_k e4m3(q[rows[i], k]) * e4m3(qW[n, k]): every
 * e4m3 value is an integer multiple of 2^-9 below 2^9 in magnitude, so each product is a multiple
 * of 2^-18 below 2^18, and a sum of at most 2^16 of them is a multiple of 2^-18 below 2^34: 52
 * significant bits, which fp64 holds exactly in any order.  absacc[i, n] = sum_k |product| bounds
 * the error of any fp32 accumulation.  Returns 1 (and computes nothing) for K > 65536, or when a
 * NaN code is present. */
int wql_oracle_fp8_acc(const uint8_t* q, const uint8_t* qW, int K, int N, const int64_t* rows,
                       int nrows, double* acc, double* absacc) {
  if (K > 65536) return 1;
  float* wdec = (float*)malloc(sizeof(float) * (size_t)N * K);
  int bad = 0;
  for (size_t i = 0; i < (size_t)N * K; ++i) {
    wdec[i] = wql_oracle_e4m3_to_float(qW[i]);
    if (isnan(wdec[i])) bad = 1;
  }
  for (int i = 0; i < nrows && !bad; ++i)
    for (int k = 0; k < K; ++k)
      if ((q[(size_t)rows[i] * K + k] & 0x7fu) == 0x7fu) bad = 1;
  if (bad) {
    free(wdec);
    return 1;
  }
#pragma omp parallel for schedule(static)
  for (int i = 0; i < nrows; ++i) {
    const uint8_t* a = q + (size_t)rows[i] * K;
    double* xa = (double*)malloc(sizeof(double) * (size_t)K);
    for (int k = 0; k < K; ++k) xa[k] = (double)wql_oracle_e4m3_to_float(a[k]);
    for (int n = 0; n < N; ++n) {
      const float* b = wdec + (size_t)n * K;
      double s = 0.0, t = 0.0;
      for (int k = 0; k < K; ++k) {
        const double p = xa[k] * (double)b[k];
        s += p;
        t += fabs(p);
      }
      acc[(size_t)i * N + n] = s;
      absacc[(size_t)i * N + n] = t;
    }
    free(xa);
  }
  free(wdec);
  return 0;
}

/* The fp8 GEMM's epilogue in fp64, without rounding: ((acc * xs_i) * ws_n + bias_n) + residual_in,
 * the terms of the int8 epilogue (a NULL bias or residual is left out). */
void wql_oracle_fp8_epilogue_f64(const double* acc, const float* xs, const float* ws,
                                 const uint16_t* bias, const uint16_t* residual, int nrows, int N,
                                 double* y) {
  for (int i = 0; i < nrows; ++i)
    for (int n = 0; n < N; ++n) {
      double u = acc[(size_t)i * N + n] * (double)xs[i] * (double)ws[n];
      if (bias) u += (double)wql_oracle_half_to_float(bias[n]);
      if (residual) u += (double)wql_oracle_half_to_float(residual[(size_t)i * N + n]);
      y[(size_t)i * N + n] = u;
    }
}

/* ---------------------------------------------------------------------------------------
 * [FastLLM] section 2: the gate and up projections of an MLP run as one fused GEMM, followed by
 * SiLU(gate) * up.  Reading: the fused weight interleaves the two projections by output channel
 * (channel 2j = gate j, channel 2j + 1 = up j), and out[r, j] = silu(y[r, 2j]) * y[r, 2j + 1] with
 * silu(g) = g / (1 + exp(-g)).  Here in fp64 on the fp64 GEMM output, without rounding (the
 * reference the fused kernel is compared with, within the W4A16 tolerance).
 * ------------------------------------------------------------------------------------- */
void wql_oracle_silu_mul_f64(const double* y, int64_t rows, int N, double* out) {
  const int J = N / 2;
  for (int64_t r = 0; r < rows; ++r)
    for (int j = 0; j < J; ++j) {
      const double g = y[r * N + 2 * j], u = y[r * N + 2 * j + 1];
      out[r * J + j] = g / (1.0 + exp(-g)) * u;
    }
}

/* ---------------------------------------------------------------------------------------
 * [FastLLM] section 5.2: the KV cache quantised from fp16 to int8 in groups of 128, with the
 * dequantisation done when the cache is read.  The page fixes the width (int8) and the group size
 * (128) only.  Reading: a group is 128 consecutive channels of one row (one token's K or V
 * vector), symmetric like the pages' per-token int8 -- s = absmax / 127 in fp32 (1.0 for an
 * all-zero group), q = clamp(rint(x / s), -128, 127) -- and the cache entry is x' = fp16(q * s).
 * kv is [rows, D] fp16 with D a multiple of 128; q is [rows, D]; scales is [rows, D / 128].
 * ------------------------------------------------------------------------------------- */
void wql_oracle_kv_quant_i8(const uint16_t* kv, int64_t rows, int D, int8_t* q, float* scales) {
  const int groups = D / 128;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int g = 0; g < groups; ++g) {
      const uint16_t* x = kv + r * D + (int64_t)g * 128;
      float amax = 0.0f;
      for (int k = 0; k < 128; ++k) {
        float a = fabsf(wql_oracle_half_to_float(x[k]));
        if (a > amax) amax = a;
      }
      float s = amax / 127.0f;
      if (amax == 0.0f) s = 1.0f;
      scales[r * groups + g] = s;
      for (int k = 0; k < 128; ++k)
        q[r * D + (int64_t)g * 128 + k] = (int8_t)clamp_rint(wql_oracle_half_to_float(x[k]) / s, -128.0f, 127.0f);
    }
}

void wql_oracle_kv_dequant_i8(const int8_t* q, const float* scales, int64_t rows, int D, uint16_t* out) {
  const int groups = D / 128;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int k = 0; k < D; ++k) {
      float v = (float)q[r * D + k] * scales[r * groups + k / 128];
      out[r * D + k] = wql_oracle_float_to_half(v);
    }
}

/* Off-path: symmetric per-tensor int4 as printed in [AWQ] section 2 (scale = max|w| / 7.5,
 * codes rounded and clipped to [-7, 7]).  Kept only to check the page's printed example. */
float wql_oracle_sym_int4_per_tensor(const float* w, int64_t n, int8_t* q) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(w[i]);
    if (a > amax) amax = a;
  }
  float scale = amax / 7.5f;
  for (int64_t i = 0; i < n; ++i) q[i] = (int8_t)clamp_rint(w[i] / scale, -7.0f, 7.0f);
  return scale;
}
