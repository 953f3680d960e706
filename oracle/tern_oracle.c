/*
 * Ternary-weight linear layer: CPU ORACLE.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously-correct definition that the CUDA
 * path is checked against.  Only tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or constant
 * with the CUDA library, and never calls it.
 *
 * What it computes (all citations name a web page and a section on it):
 *
 *  - Ternary weights w in {-1, 0, +1} with one fp16 scale per 128 consecutive
 *    weights along K ("NInfer sm_89 fork" write-up,
 *    section 9 "why NInfer is fast", item 2 "ternary weights": codes plus one
 *    FP16 scale per 128 weights).
 *
 *  - 2-bit packing.  The pages pack base-3 trits five to a byte; this layer
 *    stores each weight in 2 bits as sign and magnitude: a "nonzero" bit
 *    |w| and a "negative" bit.  Byte b of row n (bytes in little-endian order
 *    within the uint32 words, so word n*(K/16) + k/16) holds the four weights
 *    k = 4b + i, i = 0..3; weight i has its nonzero bit at bit P[i] and its
 *    negative bit at bit P[i] + 2 of the byte, with P = {0, 1, 4, 5}:
 *        (nz, neg) = (0, 0) -> 0,  (1, 0) -> +1,  (1, 1) -> -1,
 *        (0, 1) -> invalid.
 *    (Each nibble therefore reads [nz_lo, nz_hi, neg_lo, neg_hi].)
 *
 *  - bf16 rungs (T <= 16):  y[t,n] = sum_g s[n,g] * sum_{k in g} w[n,k] x[t,k]
 *    accumulated in fp64 here; m[t,n] = sum_k |s w x| is the tolerance scale.
 *
 *  - s8 rung (T >= 17): per token a = max_k |x|, xs = a / 127 (fp32),
 *    q = clamp(rint(x / xs), -127, 127) with round-to-nearest-even, then
 *    acc[t,n,g] = sum_{k in g} q w exactly in integers and
 *    y = xs * sum_g s * acc (fp64 here).  Int8 activations x ternary-as-int8
 *    weights with int32 accumulation is the "s8" prefill rung of the
 *    "ninfer-perf-tuning" skill page, section 2 rung map
 *    and section 4 numeric gate; per-token absmax/127 with round-to-nearest-even
 *    is the reading of "quantised per token to int8".
 *
 *  - base-3 packing, five weights per byte ("NInfer sm_89 fork" write-up,
 *    section 9, item 2: base-3 codes five to a byte with one FP16 scale per
 *    128 weights, 1.75 bits per weight on average).  Each 128-weight group of
 *    a row takes ceil(128/5) = 26 bytes; with its fp16 scale that is 28 bytes
 *    per 128 weights, exactly the 1.75 bits the page gives.  Byte j of group
 *    g of row n is P[(n*G + g)*26 + j] and holds the weights
 *    k = 128g + 5j + i, i = 0..4, as the base-3 number
 *        byte = sum_i (w_i + 1) * 3^i          (0..242),
 *    so the first weight is the least significant digit.  The last byte of a
 *    group holds three weights; its digits 3 and 4 are padding written as
 *    weight 0 and ignored on reading.  Bytes 243..255 are invalid.  The
 *    scales stay in their own [N][K/128] fp16 array, as for the 2-bit code.
 *
 *  - Hadamard rotation of the activations in 1024-wide blocks, applied before
 *    the layer ("NInfer sm_89 fork" write-up, section 9, item 2: the original
 *    model's Hadamard rotation is fused into the activation quantisation; the
 *    "ninfer-perf-tuning" skill page, section 6 budget table: the rotation
 *    works on (1024-block, token) pairs of bf16 activations):
 *        xr[t][bB + i] = B^(-1/2) * sum_j (-1)^popcount(i & j) x[t][bB + j]
 *    in fp64 (exact for B = 1024, whose scale is 1/32, while the inputs' bits
 *    span under 43 binary places), then rounded once to bf16, nearest-even.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - the 2-bit code is sign-magnitude with the bit order above;
 *  - the base-3 byte is a plain base-3 integer, least significant digit
 *    first, 26 bytes per group with padding digits for weight 0;
 *  - the rotation matrix is the Sylvester (natural-order) Hadamard matrix,
 *    orthonormalised by B^(-1/2); its output is rounded to bf16 once, and the
 *    layer then runs on the rounded values exactly as without rotation;
 *  - an invalid code (the 2-bit pair (0, 1), a base-3 byte above 242) reads
 *    as weight 0 in every definition here, as the library documents for its
 *    kernels, and is counted by the unpack functions;
 *  - the quantiser divides by xs = a/127 in IEEE fp32 and clamps to +-127;
 *  - a token whose absmax is 0 gets xs = 0 and q = 0.
 *
 * Build: plain C11, no fast-math, optional OpenMP over output rows.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- scalar conversions (exact widenings) ------------------------------ */

/* bf16 -> fp32 is the upper 16 bits of an fp32: exact. */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* IEEE binary16 -> double, written out from the format definition:
 * sign(1) exponent(5, bias 15) fraction(10); subnormals when exponent == 0. */
static double f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* f * 2^-10 * 2^-14 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp(1.0 + (double)f / 1024.0, e - 15);
  return sign ? -v : v;
}

/* ---- packing ------------------------------------------------------------ */

/* Bit position of the nonzero bit of weight i (0..3) within its byte; the
 * negative bit sits two places higher. */
static const int kNzBit[4] = {0, 1, 4, 5};

/* Weight (n, k) from the packed matrix; returns 2 for the invalid pair
 * (nz = 0, neg = 1) so that callers can count it. */
static int unpack_one(const uint32_t* wp, int K, int n, int k) {
  uint32_t word = wp[(size_t)n * (size_t)(K / 16) + (size_t)(k / 16)];
  uint32_t byte = (word >> (8 * ((k % 16) / 4))) & 0xffu;
  int p = kNzBit[k % 4];
  int nz = (int)((byte >> p) & 1u);
  int neg = (int)((byte >> (p + 2)) & 1u);
  if (!nz) return neg ? 2 : 0;
  return neg ? -1 : 1;
}

/* W [N][K] int8 in {-1,0,1} -> packed [N][K/16] u32.  Values outside
 * {-1,0,1} are stored as 0 and counted; the count is returned. */
long tern_oracle_pack(const int8_t* W, int K, int N, uint32_t* wp) {
  long bad = 0;
  size_t words = (size_t)N * (size_t)(K / 16);
  memset(wp, 0, words * sizeof(uint32_t));
  for (int n = 0; n < N; ++n) {
    for (int k = 0; k < K; ++k) {
      int w = W[(size_t)n * K + k];
      if (w < -1 || w > 1) {
        ++bad;
        w = 0;
      }
      uint32_t nz = (w != 0), neg = (w < 0);
      int p = 8 * ((k % 16) / 4) + kNzBit[k % 4];
      wp[(size_t)n * (K / 16) + k / 16] |= (nz << p) | (neg << (p + 2));
    }
  }
  return bad;
}

/* packed -> W [N][K] int8; invalid pairs become 0 and are counted. */
long tern_oracle_unpack(const uint32_t* wp, int K, int N, int8_t* W) {
  long bad = 0;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      int w = unpack_one(wp, K, n, k);
      if (w == 2) {
        ++bad;
        w = 0;
      }
      W[(size_t)n * K + k] = (int8_t)w;
    }
  return bad;
}

/* ---- base-3 packing: five weights per byte ------------------------------- */

#define T5_GROUP_BYTES 26 /* ceil(128 / 5) */

/* Weight (n, k) from a base-3 packed matrix; 2 for an invalid byte. */
static int unpack_one_t5(const uint8_t* p, int K, int n, int k) {
  int G = K / 128, r = k % 128;
  unsigned v = p[((size_t)n * G + k / 128) * T5_GROUP_BYTES + r / 5];
  if (v > 242u) return 2;
  for (int i = 0; i < r % 5; ++i) v /= 3u;
  return (int)(v % 3u) - 1;
}

/* W [N][K] int8 in {-1,0,1} -> base-3 bytes [N][K/128][26].  Values outside
 * {-1,0,1} are stored as 0 and counted; the count is returned. */
long tern_oracle_pack_t5(const int8_t* W, int K, int N, uint8_t* p) {
  long bad = 0;
  int G = K / 128;
  for (int n = 0; n < N; ++n)
    for (int g = 0; g < G; ++g)
      for (int j = 0; j < T5_GROUP_BYTES; ++j) {
        unsigned v = 0, place = 1;
        for (int i = 0; i < 5; ++i, place *= 3u) {
          int r = 5 * j + i, w = 0;
          if (r < 128) {
            w = W[(size_t)n * K + (size_t)g * 128 + r];
            if (w < -1 || w > 1) {
              ++bad;
              w = 0;
            }
          }
          v += (unsigned)(w + 1) * place;
        }
        p[((size_t)n * G + g) * T5_GROUP_BYTES + j] = (uint8_t)v;
      }
  return bad;
}

/* base-3 bytes -> W [N][K] int8; the weights of an invalid byte become 0.
 * Returns the number of invalid bytes. */
long tern_oracle_unpack_t5(const uint8_t* p, int K, int N, int8_t* W) {
  long bad = 0;
  size_t bytes = (size_t)N * (size_t)(K / 128) * T5_GROUP_BYTES;
  for (size_t b = 0; b < bytes; ++b) bad += p[b] > 242u;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      int w = unpack_one_t5(p, K, n, k);
      W[(size_t)n * K + k] = (int8_t)(w == 2 ? 0 : w);
    }
  return bad;
}

/* ---- the weight as the layer reads it ------------------------------------ */

/* Both packed formats go through one reader type, so each definition below
 * is written once.  An invalid code reads as 0. */
typedef int (*weight_reader)(const void* packed, int K, int n, int k);

static int read_2bit(const void* packed, int K, int n, int k) {
  int w = unpack_one((const uint32_t*)packed, K, n, k);
  return w == 2 ? 0 : w;
}

static int read_t5(const void* packed, int K, int n, int k) {
  int w = unpack_one_t5((const uint8_t*)packed, K, n, k);
  return w == 2 ? 0 : w;
}

/* ---- bf16 rungs: plain fp64 definition ----------------------------------- */

/* y = sum_g s[n][g] * sum_{k in g} w[n][k] * x[t][k] for one output (fp64),
 * one sequential sum in k order; *m = sum_g sum_{k in g} |s w x|. */
static double dot_f64(weight_reader rd, const void* packed,
                      const uint16_t* scales, const uint16_t* x, int K, int t,
                      int n, double* m) {
  int G = K / 128;
  double acc = 0.0, mag = 0.0;
  for (int g = 0; g < G; ++g) {
    double s = f16_to_f64(scales[(size_t)n * G + g]);
    double part = 0.0, partm = 0.0;
    for (int k = g * 128; k < (g + 1) * 128; ++k) {
      int w = rd(packed, K, n, k);
      double xv = (double)bf16_to_f32(x[(size_t)t * K + k]);
      part += (double)w * xv;
      partm += fabs((double)w * xv);
    }
    acc += s * part;
    mag += fabs(s) * partm;
  }
  *m = mag;
  return acc;
}

/* y [T][N], m [T][N] (m may be NULL); rows n are split across threads. */
static void linear_f64(weight_reader rd, const void* packed,
                       const uint16_t* scales, const uint16_t* x, int T, int K,
                       int N, double* y, double* m) {
#pragma omp parallel for schedule(dynamic, 16)
  for (int n = 0; n < N; ++n)
    for (int t = 0; t < T; ++t) {
      double mag;
      y[(size_t)t * N + n] = dot_f64(rd, packed, scales, x, K, t, n, &mag);
      if (m) m[(size_t)t * N + n] = mag;
    }
}

/* The same for a list of sampled outputs (t_idx[i], n_idx[i]). */
static void linear_f64_sampled(weight_reader rd, const void* packed,
                               const uint16_t* scales, const uint16_t* x,
                               int K, const int* t_idx, const int* n_idx,
                               long count, double* y, double* m) {
#pragma omp parallel for schedule(dynamic, 64)
  for (long i = 0; i < count; ++i) {
    double mag;
    y[i] = dot_f64(rd, packed, scales, x, K, t_idx[i], n_idx[i], &mag);
    if (m) m[i] = mag;
  }
}

/* scales: fp16 bits [N][K/128]; x: bf16 bits [T][K]; 2-bit weights
 * [N][K/16] u32 or base-3 weights [N][K/128][26] bytes. */
void tern_oracle_linear_f64(const uint32_t* wp, const uint16_t* scales,
                            const uint16_t* x, int T, int K, int N, double* y,
                            double* m) {
  linear_f64(read_2bit, wp, scales, x, T, K, N, y, m);
}

void tern_oracle_linear_f64_sampled(const uint32_t* wp, const uint16_t* scales,
                                    const uint16_t* x, int K, int N,
                                    const int* t_idx, const int* n_idx,
                                    long count, double* y, double* m) {
  (void)N;
  linear_f64_sampled(read_2bit, wp, scales, x, K, t_idx, n_idx, count, y, m);
}

void tern_oracle_linear_t5_f64(const uint8_t* p, const uint16_t* scales,
                               const uint16_t* x, int T, int K, int N,
                               double* y, double* m) {
  linear_f64(read_t5, p, scales, x, T, K, N, y, m);
}

void tern_oracle_linear_t5_f64_sampled(const uint8_t* p,
                                       const uint16_t* scales,
                                       const uint16_t* x, int K, int N,
                                       const int* t_idx, const int* n_idx,
                                       long count, double* y, double* m) {
  (void)N;
  linear_f64_sampled(read_t5, p, scales, x, K, t_idx, n_idx, count, y, m);
}

/* ---- s8 rung ------------------------------------------------------------- */

/* Per-token int8 quantisation, fp32 arithmetic:
 *   a  = max_k |x[t][k]|
 *   xs = a / 127.0f                       (IEEE single division)
 *   q  = clamp(rintf(x / xs), -127, 127)  (rintf: round to nearest even)
 * a == 0 gives xs = 0 and q = 0. */
void tern_oracle_quant_s8(const uint16_t* x, int T, int K, int8_t* q,
                          float* xs) {
  for (int t = 0; t < T; ++t) {
    float a = 0.0f;
    for (int k = 0; k < K; ++k) {
      float v = fabsf(bf16_to_f32(x[(size_t)t * K + k]));
      if (v > a) a = v;
    }
    float scale = a / 127.0f;
    xs[t] = scale;
    for (int k = 0; k < K; ++k) {
      float r = 0.0f;
      if (a > 0.0f) {
        r = rintf(bf16_to_f32(x[(size_t)t * K + k]) / scale);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
      }
      q[(size_t)t * K + k] = (int8_t)r;
    }
  }
}

/* Exact per-group integer accumulators and the fp64 output for one output:
 *   acc[g] = sum_{k in g} q[t][k] * w[n][k]          (int64, exact)
 *   y      = xs[t] * sum_g s[n][g] * acc[g]          (fp64)
 *   *m     = xs[t] * sum_g |s[n][g] * acc[g]|        (tolerance scale)
 * acc may be NULL. */
static double dot_s8(weight_reader rd, const void* packed,
                     const uint16_t* scales, const int8_t* q, const float* xs,
                     int K, int t, int n, int64_t* acc, double* m) {
  int G = K / 128;
  double sum = 0.0, mag = 0.0;
  for (int g = 0; g < G; ++g) {
    int64_t a = 0;
    for (int k = g * 128; k < (g + 1) * 128; ++k)
      a += (int64_t)q[(size_t)t * K + k] * (int64_t)rd(packed, K, n, k);
    if (acc) acc[g] = a;
    double s = f16_to_f64(scales[(size_t)n * G + g]);
    sum += s * (double)a;
    mag += fabs(s * (double)a);
  }
  *m = fabs((double)xs[t]) * mag;
  return (double)xs[t] * sum;
}

/* y [T][N], acc [T][N][G], m [T][N]; acc and m may be NULL. */
static void linear_s8(weight_reader rd, const void* packed,
                      const uint16_t* scales, const int8_t* q, const float* xs,
                      int T, int K, int N, int64_t* acc, double* y, double* m) {
  int G = K / 128;
#pragma omp parallel for schedule(dynamic, 16)
  for (int n = 0; n < N; ++n)
    for (int t = 0; t < T; ++t) {
      double mag;
      size_t o = (size_t)t * N + n;
      y[o] = dot_s8(rd, packed, scales, q, xs, K, t, n, acc ? acc + o * G : NULL,
                    &mag);
      if (m) m[o] = mag;
    }
}

/* The same for sampled outputs; acc is [count][G]. */
static void linear_s8_sampled(weight_reader rd, const void* packed,
                              const uint16_t* scales, const int8_t* q,
                              const float* xs, int K, const int* t_idx,
                              const int* n_idx, long count, int64_t* acc,
                              double* y, double* m) {
  int G = K / 128;
#pragma omp parallel for schedule(dynamic, 64)
  for (long i = 0; i < count; ++i) {
    double mag;
    y[i] = dot_s8(rd, packed, scales, q, xs, K, t_idx[i], n_idx[i],
                  acc ? acc + (size_t)i * G : NULL, &mag);
    if (m) m[i] = mag;
  }
}

void tern_oracle_linear_s8(const uint32_t* wp, const uint16_t* scales,
                           const int8_t* q, const float* xs, int T, int K,
                           int N, int64_t* acc, double* y, double* m) {
  linear_s8(read_2bit, wp, scales, q, xs, T, K, N, acc, y, m);
}

void tern_oracle_linear_s8_sampled(const uint32_t* wp, const uint16_t* scales,
                                   const int8_t* q, const float* xs, int K,
                                   int N, const int* t_idx, const int* n_idx,
                                   long count, int64_t* acc, double* y,
                                   double* m) {
  (void)N;
  linear_s8_sampled(read_2bit, wp, scales, q, xs, K, t_idx, n_idx, count, acc,
                    y, m);
}

void tern_oracle_linear_t5_s8(const uint8_t* p, const uint16_t* scales,
                              const int8_t* q, const float* xs, int T, int K,
                              int N, int64_t* acc, double* y, double* m) {
  linear_s8(read_t5, p, scales, q, xs, T, K, N, acc, y, m);
}

void tern_oracle_linear_t5_s8_sampled(const uint8_t* p, const uint16_t* scales,
                                      const int8_t* q, const float* xs, int K,
                                      int N, const int* t_idx,
                                      const int* n_idx, long count,
                                      int64_t* acc, double* y, double* m) {
  (void)N;
  linear_s8_sampled(read_t5, p, scales, q, xs, K, t_idx, n_idx, count, acc, y,
                    m);
}

/* ---- Hadamard rotation of the activations --------------------------------- */

/* fp64 -> bf16 bits, round to nearest, ties to even, in one step from the
 * double (no intermediate fp32).  From the format: sign, 8 exponent bits
 * (bias 127), 7 fraction bits; normal values have 8 significant bits, values
 * below 2^-126 are subnormal with quantum 2^-133; magnitudes that round to
 * 2^128 or above become infinity. */
static uint16_t f64_to_bf16(double d) {
  if (isnan(d)) return 0x7FC0;
  uint16_t sign = signbit(d) ? 0x8000 : 0;
  double a = fabs(d);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e); /* a = m 2^e, 0.5 <= m < 1: the leading bit is worth 2^(e-1) */
  int q = e - 8; /* quantum of an 8-significant-bit value */
  if (q < -133) q = -133;
  double r = rint(ldexp(a, -q)); /* integer multiple of the quantum, RNE */
  double v = ldexp(r, q);
  if (v >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  float f = (float)v; /* exact: v is a bf16 value */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

void tern_oracle_f64_to_bf16(const double* v, long n, uint16_t* out) {
  for (long i = 0; i < n; ++i) out[i] = f64_to_bf16(v[i]);
}

/* Popcount parity of i & j: the sign of entry (i, j) of the Sylvester
 * Hadamard matrix is (-1)^parity. */
static int hadamard_sign(int i, int j) {
  unsigned v = (unsigned)(i & j);
  int p = 0;
  while (v) {
    p ^= 1;
    v &= v - 1u;
  }
  return p ? -1 : 1;
}

/* x: bf16 bits [T][K]; B: block width, a power of two dividing K.
 *   exact[t][k] = B^(-1/2) * sum over the block of k of sign * x   (fp64)
 *   xr[t][k]    = bf16 of exact[t][k]
 * Either output may be NULL.  The sum over j runs in j order. */
void tern_oracle_rotate(const uint16_t* x, int T, int K, int B, double* exact,
                        uint16_t* xr) {
  double norm = 1.0 / sqrt((double)B);
#pragma omp parallel for collapse(2) schedule(static)
  for (int t = 0; t < T; ++t)
    for (int b = 0; b < K / B; ++b)
      for (int i = 0; i < B; ++i) {
        double acc = 0.0;
        for (int j = 0; j < B; ++j)
          acc += (double)hadamard_sign(i, j) *
                 (double)bf16_to_f32(x[(size_t)t * K + (size_t)b * B + j]);
        double v = acc * norm;
        size_t o = (size_t)t * K + (size_t)b * B + i;
        if (exact) exact[o] = v;
        if (xr) xr[o] = f64_to_bf16(v);
      }
}

int tern_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
