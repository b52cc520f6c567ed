/*
 * nf4_oracle.c -- plain CPU oracle for NF4 weight-quantized projections.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg load this library.  The product
 * library (the CUDA path) never includes, links or calls anything here, and
 * this file includes nothing from the product.
 *
 * Source: "Decode V2 -- resident executor" (deep-fold docs/decode-v2.md),
 *   section 2 "Synthetic models" (linears are NF4, dims are multiples of the
 *   64-weight NF4 group), section 3 "CPU oracle" (decode_nf4 then matmul;
 *   SwiGLU = silu(gate) * up with SiLU applied to the full gate sum; greedy id =
 *   argmax of the logits), section 6 "Linear primitive" (FP32 LUT x scale x x;
 *   N=1 takes a [K] view; o/down add a residual into y; prefill chunks of 32).
 * Gate/up rows interleaved in one matrix: "gizai:tensor/lazy", method
 *   Lazy.gluIn (output column c = silu of row 2c times row 2c + 1).
 * Argmax tie rule: golang.design/x/accel/tensor, "func Argmax", paragraph
 *   "Ties go to the lowest index".
 * bf16 -> f32 widening is exact: same page, "func Cast", "bf16 widens and does
 *   not narrow".
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *  - codebook: the 16 NormalFloat levels of the QLoRA construction (Dettmers et
 *    al. 2023, section 3): quantiles of N(0,1) at evenly spaced probabilities,
 *    8 on the positive side, 7 on the negative side, plus an exact 0, divided by
 *    the largest, sorted ascending.  Computed here in float64 with an inverse
 *    normal CDF found by bisection on Phi(z) = erfc(-z/sqrt 2)/2, then rounded
 *    once to fp32.
 *  - encoder: scale = absmax of the 64-block (fp32, exact); an all-zero block
 *    gets scale 0 and code 7 (the exact-zero level); otherwise each weight takes
 *    the level nearest to w/scale in exact arithmetic, ties to the lower index.
 *  - layout: codes[M][K/2], byte j of a row holds k=2j in bits 0-3 and k=2j+1
 *    in bits 4-7; scales[M][K/64] fp32; rows K-contiguous.
 *  - dequant: W_hat[m][k] = fp32(cb[code] * scale) (one fp32 rounding).
 *  - sums: float64, k ascending; epilogues in float64 from the float64 sums,
 *    rounded once to the output type (round to nearest even).
 *  - prefill chunk: the weight is dequantized to bf16 (RN of the fp32 W_hat)
 *    before the product, as the chunk's tensor-core path does; the sum is float64.
 *
 * No blocking, fusion or reordering beyond these definitions.
 *
 * The nf4o_* functions take per-row selections and return float64 values (and
 * the magnitudes S) for the tests; the nf4_ref_* functions at the end take the
 * library's own argument lists with host pointers and return its output types.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define NF4O_OK 0
#define NF4O_EINVAL (-1)

/* x / X element types, same numbering as the public API uses for activations. */
#define NF4O_F32 0
#define NF4O_BF16 1

/* ---------------------------------------------------------------- codebook */

/* Phi(z) for the standard normal distribution, through libm's erfc. */
static double std_normal_cdf(double z) { return 0.5 * erfc(-z / sqrt(2.0)); }

/* Inverse of Phi by bisection: the z with Phi(z) = p, to double resolution. */
static double std_normal_quantile(double p) {
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 2000; ++it) {
    double mid = 0.5 * (lo + hi);
    if (mid == lo || mid == hi) break;
    if (std_normal_cdf(mid) < p)
      lo = mid;
    else
      hi = mid;
  }
  return 0.5 * (lo + hi);
}

/* The 16 NF4 levels, ascending, fp32.  cb[0] = -1, cb[7] = 0, cb[15] = +1. */
int nf4o_codebook(float cb[16]) {
  const double delta = 0.5 * (1.0 / 32.0 + 1.0 / 30.0);
  double v[16];
  int n = 0;
  /* 8 levels on the positive side: probabilities from 1-delta down towards 1/2 */
  for (int j = 0; j < 8; ++j) v[n++] = std_normal_quantile(1.0 - delta - j * (0.5 - delta) / 8.0);
  /* 7 levels on the negative side: probabilities from delta up towards 1/2 */
  for (int j = 0; j < 7; ++j) v[n++] = std_normal_quantile(delta + j * (0.5 - delta) / 7.0);
  v[n++] = 0.0;
  const double top = std_normal_quantile(1.0 - delta);
  for (int i = 0; i < 16; ++i) v[i] /= top;
  /* insertion sort, ascending */
  for (int i = 1; i < 16; ++i) {
    double t = v[i];
    int j = i - 1;
    while (j >= 0 && v[j] > t) {
      v[j + 1] = v[j];
      --j;
    }
    v[j + 1] = t;
  }
  for (int i = 0; i < 16; ++i) cb[i] = (float)v[i];
  return NF4O_OK;
}

/* ------------------------------------------------------------- bit helpers */

static float bf16_bits_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round a double to the nearest bf16 (ties to even); returns the bits. */
static uint16_t f64_to_bf16_bits(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
  /* bf16 keeps 8 significant bits; its smallest normal is 2^-126 and its
   * subnormals step by 2^-133. */
  int q = e - 8;
  if (q < -133) q = -133;
  double r = rint(ldexp(a, -q)); /* default rounding mode: to nearest even */
  double rv = ldexp(r, q);
  /* re-encode rv: exactly representable in bf16 unless it rounded up to 2^128 */
  if (rv > 3.3895313892515355e38 /* largest finite bf16, (2 - 2^-7) * 2^127 */) return sign | 0x7F80;
  float f = (float)rv; /* exact: rv has <= 8 significant bits within fp32 range */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* Round an fp32 to the nearest bf16 (ties to even); returns the value as fp32. */
static float f32_round_bf16(float f) { return bf16_bits_to_f32(f64_to_bf16_bits((double)f)); }

static double load_x(const void* x, int xt, int64_t k) {
  if (xt == NF4O_BF16) return (double)bf16_bits_to_f32(((const uint16_t*)x)[k]);
  return (double)((const float*)x)[k];
}

static int code_at(const uint8_t* codes, int64_t K, int64_t m, int64_t k) {
  uint8_t byte = codes[m * (K / 2) + k / 2];
  return (k & 1) ? (byte >> 4) : (byte & 0x0F);
}

static float what_at(const float cb[16], const uint8_t* codes, const float* scales, int64_t K, int64_t m,
                     int64_t k) {
  float c = cb[code_at(codes, K, m, k)];
  float s = scales[m * (K / 64) + k / 64];
  return c * s; /* one fp32 rounding */
}

static int shape_ok(int64_t M, int64_t K) { return M >= 1 && K >= 64 && K % 64 == 0; }

/* ----------------------------------------------------------------- encoder */

/*
 * Nearest level to w/s with ties to the lower index, decided exactly.
 * The tie point between levels i and i+1 is mid_i = (cb[i] + cb[i+1]) / 2.
 * w/s > mid_i  <=>  w > mid_i * s  for s > 0, and both mid_i and mid_i * s are
 * exact in float64 (cb values carry 24 significant bits, their sums at most 26,
 * the product with a 24-bit scale at most 50), so the comparison below is the
 * exact-arithmetic one.  The code is the number of tie points strictly below.
 */
static int nearest_code(const float cb[16], float w, float s) {
  int code = 0;
  for (int i = 0; i < 15; ++i) {
    double mid = ((double)cb[i] + (double)cb[i + 1]) / 2.0;
    if ((double)w > mid * (double)s) ++code;
  }
  return code;
}

int nf4o_quantize(const float* W, int64_t M, int64_t K, uint8_t* codes, float* scales) {
  if (!shape_ok(M, K) || !W || !codes || !scales) return NF4O_EINVAL;
  float cb[16];
  nf4o_codebook(cb);
  const int64_t nb = K / 64;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* w = W + m * K + b * 64;
      float s = 0.0f;
      for (int i = 0; i < 64; ++i) {
        if (!isfinite(w[i])) return NF4O_EINVAL;
        float a = fabsf(w[i]);
        if (a > s) s = a;
      }
      scales[m * nb + b] = s;
      uint8_t* out = codes + m * (K / 2) + b * 32;
      for (int j = 0; j < 32; ++j) {
        int lo = (s == 0.0f) ? 7 : nearest_code(cb, w[2 * j], s);
        int hi = (s == 0.0f) ? 7 : nearest_code(cb, w[2 * j + 1], s);
        out[j] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
  return NF4O_OK;
}

/* ------------------------------------------------------------------ decode */

int nf4o_dequant(const uint8_t* codes, const float* scales, int64_t M, int64_t K, float* W_hat) {
  if (!shape_ok(M, K) || !codes || !scales || !W_hat) return NF4O_EINVAL;
  float cb[16];
  nf4o_codebook(cb);
  for (int64_t m = 0; m < M; ++m)
    for (int64_t k = 0; k < K; ++k) W_hat[m * K + k] = what_at(cb, codes, scales, K, m, k);
  return NF4O_OK;
}

/* --------------------------------------------------------------- N=1 GEMV */

/*
 * y[i] = sum_k W_hat[m][k] * x[k] in float64, k ascending, for m = rows[i]
 * (all rows in order when rows is NULL).  S[i] = sum_k |W_hat[m][k] * x[k]|,
 * the per-row magnitude the tolerance is stated against.  Either output may be
 * NULL.
 */
int nf4o_gemv(const uint8_t* codes, const float* scales, int64_t M, int64_t K, const void* x, int xt,
              const int64_t* rows, int64_t nrows, double* y, double* S) {
  if (!shape_ok(M, K) || !codes || !scales || !x) return NF4O_EINVAL;
  if (xt != NF4O_F32 && xt != NF4O_BF16) return NF4O_EINVAL;
  if (!rows) nrows = M;
  float cb[16];
  nf4o_codebook(cb);
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = rows ? rows[i] : i;
    if (m < 0 || m >= M) return NF4O_EINVAL;
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double t = (double)what_at(cb, codes, scales, K, m, k) * load_x(x, xt, k);
      acc += t;
      mag += fabs(t);
    }
    if (y) y[i] = acc;
    if (S) S[i] = mag;
  }
  return NF4O_OK;
}

/* y = W x + r, float64 sum plus the residual, rounded once to fp32. */
int nf4o_gemv_residual(const uint8_t* codes, const float* scales, int64_t M, int64_t K, const void* x,
                       int xt, const float* r, const int64_t* rows, int64_t nrows, double* y_f64,
                       float* y_f32) {
  if (!r) return NF4O_EINVAL;
  if (!rows) nrows = M;
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = rows ? rows[i] : i;
    double acc;
    int st = nf4o_gemv(codes, scales, M, K, x, xt, &m, 1, &acc, NULL);
    if (st) return st;
    double v = acc + (double)r[m];
    if (y_f64) y_f64[i] = v;
    if (y_f32) y_f32[i] = (float)v;
  }
  return NF4O_OK;
}

/*
 * Fused q/k/v projection ("Decode V2 -- resident executor", section 6: one
 * grid over q.M + k.M + v.M rows sharing x, the q/k/v bias added in the same
 * kernel).  The row space is the three matrices' rows in the order q, k, v;
 * for row r of matrix p:
 *   y = sum_k W_hat_p[r][k] * x[k] + b_p[r]      (float64, k ascending)
 *   S = sum_k |W_hat_p[r][k] * x[k]| + |b_p[r]|
 * b_p NULL means no bias for matrix p.  rows[] index the concatenated row
 * space (all rows in order when rows is NULL); y or S may be NULL.
 */
int nf4o_gemv_qkv(const uint8_t* const codes[3], const float* const scales[3], const float* const bias[3],
                  const int64_t M[3], int64_t K, const void* x, int xt, const int64_t* rows, int64_t nrows,
                  double* y, double* S) {
  if (!codes || !scales || !bias || !M) return NF4O_EINVAL;
  const int64_t total = M[0] + M[1] + M[2];
  if (!rows) nrows = total;
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t r = rows ? rows[i] : i;
    if (r < 0 || r >= total) return NF4O_EINVAL;
    int p = 0;
    while (r >= M[p]) {
      r -= M[p];
      ++p;
    }
    double acc, mag;
    int st = nf4o_gemv(codes[p], scales[p], M[p], K, x, xt, &r, 1, &acc, &mag);
    if (st) return st;
    const double b = bias[p] ? (double)bias[p][r] : 0.0;
    if (y) y[i] = acc + b;
    if (S) S[i] = mag + fabs(b);
  }
  return NF4O_OK;
}

/*
 * Embedding rows kept as NF4 ("Decode V2 -- resident executor", section 10:
 * the embedding stays as NF4 rows, gathered and dequantized into the arena,
 * with no dense [vocab, hidden] table).  For i < n:
 *   out_f32[i][k]  = W_hat[ids[i]][k]   (level x scale, one fp32 rounding)
 *   out_bf16[i][k] = that value rounded to bf16 (nearest even)
 * Rows whose id lies outside [0, V) are written as zeros and counted in *bad.
 * Any output may be NULL.
 */
int nf4o_dequant_rows(const uint8_t* codes, const float* scales, int64_t V, int64_t K, const int64_t* ids,
                      int64_t n, float* out_f32, uint16_t* out_bf16, int64_t* bad) {
  if (!shape_ok(V, K) || !codes || !scales || (n > 0 && !ids) || n < 0) return NF4O_EINVAL;
  float cb[16];
  nf4o_codebook(cb);
  int64_t nbad = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t m = ids[i];
    const int ok = m >= 0 && m < V;
    nbad += !ok;
    for (int64_t k = 0; k < K; ++k) {
      const float w = ok ? what_at(cb, codes, scales, K, m, k) : 0.0f;
      if (out_f32) out_f32[i * K + k] = w;
      if (out_bf16) out_bf16[i * K + k] = f64_to_bf16_bits((double)w);
    }
  }
  if (bad) *bad = nbad;
  return NF4O_OK;
}

/* silu(z) = z / (1 + e^-z), float64 */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * out[i] = silu(g_m) * u_m with g = Wg x and u = Wu x (float64 sums over the
 * full K), rounded once to bf16.  out_f64 gets the unrounded value, out_bf16
 * the rounded bits, g/u the float64 sums.  Any output may be NULL.
 */
int nf4o_gemv_swiglu(const uint8_t* g_codes, const float* g_scales, const uint8_t* u_codes,
                     const float* u_scales, int64_t M, int64_t K, const void* x, int xt,
                     const int64_t* rows, int64_t nrows, double* out_f64, uint16_t* out_bf16,
                     double* g, double* u) {
  if (!rows) nrows = M;
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = rows ? rows[i] : i;
    double gs, us;
    int st = nf4o_gemv(g_codes, g_scales, M, K, x, xt, &m, 1, &gs, NULL);
    if (st) return st;
    st = nf4o_gemv(u_codes, u_scales, M, K, x, xt, &m, 1, &us, NULL);
    if (st) return st;
    double v = silu(gs) * us;
    if (out_f64) out_f64[i] = v;
    if (out_bf16) out_bf16[i] = f64_to_bf16_bits(v);
    if (g) g[i] = gs;
    if (u) u[i] = us;
  }
  return NF4O_OK;
}

/*
 * SwiGLU over one matrix whose rows alternate gate and up ("gizai:tensor/lazy",
 * method Lazy.gluIn: output column c is silu of product row 2c times product
 * row 2c + 1).  The matrix has M2 = 2 x outputs rows; v = W x in float64 as
 * nf4o_gemv; out[c] = silu(v[2c]) * v[2c + 1], rounded once to bf16 as
 * nf4o_gemv_swiglu.  `cols` (or all M2 / 2 outputs when NULL) selects outputs;
 * any output array may be NULL.  An odd M2 is rejected.
 */
int nf4o_gemv_glu_interleaved(const uint8_t* codes, const float* scales, int64_t M2, int64_t K, const void* x,
                              int xt, const int64_t* cols, int64_t ncols, double* out_f64, uint16_t* out_bf16,
                              double* g, double* u) {
  if (M2 < 2 || (M2 & 1)) return NF4O_EINVAL;
  const int64_t n_out = M2 / 2;
  if (!cols) ncols = n_out;
  for (int64_t i = 0; i < ncols; ++i) {
    const int64_t c = cols ? cols[i] : i;
    if (c < 0 || c >= n_out) return NF4O_EINVAL;
    int64_t rg = 2 * c, ru = 2 * c + 1;
    double gs, us;
    int st = nf4o_gemv(codes, scales, M2, K, x, xt, &rg, 1, &gs, NULL);
    if (st) return st;
    st = nf4o_gemv(codes, scales, M2, K, x, xt, &ru, 1, &us, NULL);
    if (st) return st;
    const double v = silu(gs) * us;
    if (out_f64) out_f64[i] = v;
    if (out_bf16) out_bf16[i] = f64_to_bf16_bits(v);
    if (g) g[i] = gs;
    if (u) u[i] = us;
  }
  return NF4O_OK;
}

/*
 * Greedy argmax over all M rows: logits_f64 (float64 sums, may be NULL),
 * logits_f32 (each rounded once to fp32, may be NULL) and the index of the
 * largest float64 logit, ties to the lowest index.
 */
int nf4o_gemv_argmax(const uint8_t* codes, const float* scales, int64_t M, int64_t K, const void* x,
                     int xt, double* logits_f64, float* logits_f32, int64_t* index) {
  if (!index) return NF4O_EINVAL;
  int64_t best = -1;
  double best_v = 0.0;
  for (int64_t m = 0; m < M; ++m) {
    double v;
    int st = nf4o_gemv(codes, scales, M, K, x, xt, &m, 1, &v, NULL);
    if (st) return st;
    if (logits_f64) logits_f64[m] = v;
    if (logits_f32) logits_f32[m] = (float)v;
    if (best < 0 || v > best_v) { /* strict: an equal later logit never wins */
      best = m;
      best_v = v;
    }
  }
  *index = best;
  return NF4O_OK;
}

/*
 * Prefill chunk: Y[n][m] = sum_k bf16(W_hat[m][k]) * X[n][k] in float64,
 * k ascending, for n < N and m = rows[i] (all rows when rows is NULL).
 * X is bf16 bits, [N][K] row-major.  Y is [N][nrows] (row-major over n).
 * S (may be NULL) gets sum_k |bf16(W_hat) * X| with the same layout.
 */
int nf4o_gemm_chunk(const uint8_t* codes, const float* scales, int64_t M, int64_t K, const uint16_t* X,
                    int64_t N, const int64_t* rows, int64_t nrows, double* Y, double* S) {
  if (!shape_ok(M, K) || !codes || !scales || !X || N < 1) return NF4O_EINVAL;
  if (!rows) nrows = M;
  float cb[16];
  nf4o_codebook(cb);
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t i = 0; i < nrows; ++i) {
      int64_t m = rows ? rows[i] : i;
      if (m < 0 || m >= M) return NF4O_EINVAL;
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double w = (double)f32_round_bf16(what_at(cb, codes, scales, K, m, k));
        double t = w * (double)bf16_bits_to_f32(X[n * K + k]);
        acc += t;
        mag += fabs(t);
      }
      if (Y) Y[n * nrows + i] = acc;
      if (S) S[n * nrows + i] = mag;
    }
  }
  return NF4O_OK;
}

/*
 * RMSNorm of `rows` rows of K values: y[r][k] = x[r][k] * w[k] / sqrt(ms_r + eps),
 * ms_r = (sum_k x[r][k]^2) / K.
 * Source: "Decode V2 -- resident executor", section 3 "CPU oracle" (RMSNorm is
 * x * rsqrt(mean(x^2) + eps) * w, Qwen-style, no bias) and section 2 (RMS
 * weights are bf16 [hidden]); "golang.design/x/accel/tensor", func RMSNorm
 * (each row normalized by its root mean square, scaled by a gain).
 * x fp32 [rows][K], w bf16 bits [K]; everything in float64, k ascending.
 * y_f64 (may be NULL) gets the float64 values, ms (may be NULL) the float64
 * mean squares.
 */
int nf4o_rmsnorm(const float* x, const uint16_t* w, int64_t rows, int64_t K, double eps, double* y_f64,
                 double* ms) {
  if (!x || !w || rows < 1 || K < 1 || !(eps >= 0.0)) return NF4O_EINVAL;
  for (int64_t r = 0; r < rows; ++r) {
    double ss = 0.0;
    for (int64_t k = 0; k < K; ++k) ss += (double)x[r * K + k] * (double)x[r * K + k];
    const double m = ss / (double)K;
    const double inv = 1.0 / sqrt(m + eps);
    if (ms) ms[r] = m;
    if (y_f64)
      for (int64_t k = 0; k < K; ++k) y_f64[r * K + k] = (double)x[r * K + k] * inv * (double)bf16_bits_to_f32(w[k]);
  }
  return NF4O_OK;
}

/* Rounding helpers exposed for the tests: double -> bf16 bits (RN-even). */
uint16_t nf4o_round_bf16(double v) { return f64_to_bf16_bits(v); }

/* ------------------------------------------------ the library's calls, on the host
 *
 * nf4_ref_* take the arguments of the library's calls of the same name
 * (nf4_gemv, ..., nf4_gemm_chunk, without the stream and the workspace) with
 * host pointers, and compute them as defined above: float64 sums, epilogues in
 * float64, each result rounded once to the output type (fp32 by C's
 * double -> float conversion, round to nearest even; bf16 by
 * f64_to_bf16_bits).  The weight descriptor is this file's own, with the same
 * members in the same order as the library's.  Each returns 0, or -1 for an
 * invalid argument (nothing is written then for the shape checks; the others
 * may stop part way).  Activation and output dtypes: 0 = fp32, 1 = bf16.
 */
typedef struct nf4_ref_weight {
  const uint8_t* codes; /* [M][K/2] */
  const float* scales;  /* [M][K/64] */
  int64_t M;
  int64_t K;
} nf4_ref_weight;

static int ref_ok(const nf4_ref_weight* W) { return W && W->codes && W->scales && shape_ok(W->M, W->K); }

int nf4_ref_quantize(const float* W, int64_t M, int64_t K, uint8_t* codes, float* scales) {
  return nf4o_quantize(W, M, K, codes, scales);
}

int nf4_ref_gemv(const nf4_ref_weight* W, const void* x, int xt, float* y) {
  if (!ref_ok(W) || !y) return NF4O_EINVAL;
  for (int64_t m = 0; m < W->M; ++m) {
    double v;
    int st = nf4o_gemv(W->codes, W->scales, W->M, W->K, x, xt, &m, 1, &v, NULL);
    if (st) return st;
    y[m] = (float)v;
  }
  return NF4O_OK;
}

/* y may alias residual: row m's residual is read before y[m] is written. */
int nf4_ref_gemv_residual(const nf4_ref_weight* W, const void* x, int xt, const float* residual, float* y) {
  if (!ref_ok(W) || !residual || !y) return NF4O_EINVAL;
  return nf4o_gemv_residual(W->codes, W->scales, W->M, W->K, x, xt, residual, NULL, 0, NULL, y);
}

int nf4_ref_gemv_swiglu(const nf4_ref_weight* Wg, const nf4_ref_weight* Wu, const void* x, int xt, uint16_t* out) {
  if (!ref_ok(Wg) || !ref_ok(Wu) || Wg->M != Wu->M || Wg->K != Wu->K || !out) return NF4O_EINVAL;
  return nf4o_gemv_swiglu(Wg->codes, Wg->scales, Wu->codes, Wu->scales, Wg->M, Wg->K, x, xt, NULL, 0, NULL, out,
                          NULL, NULL);
}

int nf4_ref_gemv_glu_interleaved(const nf4_ref_weight* W, const void* x, int xt, uint16_t* out) {
  if (!ref_ok(W) || !out) return NF4O_EINVAL;
  return nf4o_gemv_glu_interleaved(W->codes, W->scales, W->M, W->K, x, xt, NULL, 0, NULL, out, NULL, NULL);
}

/* q/k/v: each output gets its matrix's float64 sum plus its bias (bias may be NULL). */
int nf4_ref_gemv_qkv(const nf4_ref_weight* Wq, const nf4_ref_weight* Wk, const nf4_ref_weight* Wv, const float* bq,
                     const float* bk, const float* bv, const void* x, int xt, float* q, float* k, float* v) {
  const nf4_ref_weight* W[3] = {Wq, Wk, Wv};
  const float* b[3] = {bq, bk, bv};
  float* out[3] = {q, k, v};
  for (int p = 0; p < 3; ++p)
    if (!ref_ok(W[p]) || W[p]->K != Wq->K || !out[p]) return NF4O_EINVAL;
  for (int p = 0; p < 3; ++p)
    for (int64_t m = 0; m < W[p]->M; ++m) {
      double s;
      int st = nf4o_gemv(W[p]->codes, W[p]->scales, W[p]->M, W[p]->K, x, xt, &m, 1, &s, NULL);
      if (st) return st;
      out[p][m] = (float)(s + (b[p] ? (double)b[p][m] : 0.0));
    }
  return NF4O_OK;
}

int nf4_ref_gemv_argmax(const nf4_ref_weight* W, const void* x, int xt, float* logits, int64_t* index) {
  if (!ref_ok(W) || !logits || !index) return NF4O_EINVAL;
  return nf4o_gemv_argmax(W->codes, W->scales, W->M, W->K, x, xt, NULL, logits, index);
}

/* Y[n][m], X bf16 bits [N][K]; N in [1, 32] as the library's call. */
int nf4_ref_gemm_chunk(const nf4_ref_weight* W, const uint16_t* X, int N, float* Y) {
  if (!ref_ok(W) || !X || !Y || N < 1 || N > 32) return NF4O_EINVAL;
  for (int64_t m = 0; m < W->M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double s;
      int st = nf4o_gemm_chunk(W->codes, W->scales, W->M, W->K, X + n * W->K, 1, &m, 1, &s, NULL);
      if (st) return st;
      Y[n * W->M + m] = (float)s;
    }
  return NF4O_OK;
}

/* Rows E[ids[i]] as fp32 (ot 0) or bf16 (ot 1); an id outside [0, M) gives a
 * row of zeros, as the library writes it (which also reports it). */
int nf4_ref_dequant_rows(const nf4_ref_weight* E, const int64_t* ids, int64_t n, void* out, int ot) {
  if (!ref_ok(E) || (n > 0 && (!ids || !out)) || n < 0 || (ot != NF4O_F32 && ot != NF4O_BF16)) return NF4O_EINVAL;
  int64_t bad = 0;
  return nf4o_dequant_rows(E->codes, E->scales, E->M, E->K, ids, n, ot == NF4O_F32 ? (float*)out : NULL,
                           ot == NF4O_BF16 ? (uint16_t*)out : NULL, &bad);
}

/* y fp32 (yt 0, may equal x) or bf16 (yt 1); eps widened exactly to float64. */
int nf4_ref_rmsnorm(const float* x, const uint16_t* w, int64_t rows, int64_t K, float eps, void* y, int yt) {
  if (!x || !w || !y || rows < 1 || K < 1 || !(eps >= 0.0f) || (yt != NF4O_F32 && yt != NF4O_BF16)) return NF4O_EINVAL;
  for (int64_t r = 0; r < rows; ++r) {
    double ss = 0.0;
    for (int64_t k = 0; k < K; ++k) ss += (double)x[r * K + k] * (double)x[r * K + k];
    const double inv = 1.0 / sqrt(ss / (double)K + (double)eps);
    for (int64_t k = 0; k < K; ++k) {
      const double v = (double)x[r * K + k] * inv * (double)bf16_bits_to_f32(w[k]);
      if (yt == NF4O_F32)
        ((float*)y)[r * K + k] = (float)v;
      else
        ((uint16_t*)y)[r * K + k] = f64_to_bf16_bits(v);
    }
  }
  return NF4O_OK;
}
