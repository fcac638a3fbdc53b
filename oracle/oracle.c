/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the shared-input
 * batched linear.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark load it; the product library never does.
 * It shares no source, header or table with the CUDA library.
 *
 * What it computes (oxinfer 0.0.0, src/gpu.rs):
 *   - struct `Job` doc comment: one matmul of a batch sharing the input x,
 *     y[t][n_out] = x[t][n_in] * W^T, W stored [n_out, n_in] (enum `WeightRef`
 *     doc comment).
 *   - `Backend::matmul`: every job of the batch runs over the same x, t, n_in.
 *   - enum `WeightRef`: the three storage formats Bf16 / Q8 / Q4.  The page
 *     names Q8 and Q4 without defining them; this library fixes them as
 *       Q8: symmetric int8, one fp32 scale d per 32-element block along n_in,
 *           w = d * q;
 *       Q4: symmetric signed 4-bit (two's complement nibble), two values per
 *           byte, low nibble = even element, one fp32 scale per 32-block.
 *   - bf16 weights are raw u16 bit patterns (oxinfer 0.0.1 src/drafter.rs,
 *     struct `DLayer`: weights held as `&[u16]`); widening to fp32 is the
 *     exact bit shift.
 *   - gelu_mul after the gate+up batch (oxinfer 0.0.1 src/drafter.rs,
 *     `Drafter::step`), for the fused gate+up job: at the end of this file.
 *
 * Host byte layout of one weight (one contiguous buffer):
 *   BF16: u16 w[n_out][n_in]
 *   Q8  : i8  q[n_out][n_in]    then f32 d[n_out][n_in/32] at byte n_out*n_in
 *   Q4  : u8  p[n_out][n_in/2]  then f32 d[n_out][n_in/32] at byte n_out*n_in/2
 *
 * Arithmetic:
 *   dequantised weight  = fp32(d * q): the exact product rounded once to fp32
 *                         (d*q is exact in double: 24-bit * 8-bit mantissas);
 *   y_ref[t][o]         = sum_i (double)x[t][i] * (double)w[o][i], i ascending;
 *   mag[t][o]           = sum_i |(double)x[t][i] * (double)w[o][i]|.
 * Built with -ffp-contract=off so no multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORACLE_BF16 = 0, ORACLE_Q8 = 1, ORACLE_Q4 = 2 };

/* bf16 bit pattern -> fp32: the 16 bits become the top half of the fp32 word. */
static float bf16_bits_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* fp32(d*q): the exact double product, rounded once to fp32. */
static float scaled(float d, int q) { return (float)((double)d * (double)q); }

/* Element (o, i) of a weight in the host layout above, dequantised to fp32. */
static float weight_at(int format, const uint8_t* w, int64_t n_out, int64_t n_in,
                       int64_t o, int64_t i) {
  if (format == ORACLE_BF16) {
    uint16_t b;
    memcpy(&b, w + 2 * (o * n_in + i), 2);
    return bf16_bits_to_f32(b);
  }
  int64_t n_blocks = n_in / 32;
  float d;
  if (format == ORACLE_Q8) {
    const uint8_t* scales = w + n_out * n_in;
    memcpy(&d, scales + 4 * (o * n_blocks + i / 32), 4);
    int q = (int)(int8_t)w[o * n_in + i];
    return scaled(d, q);
  }
  /* Q4 */
  const uint8_t* scales = w + n_out * (n_in / 2);
  memcpy(&d, scales + 4 * (o * n_blocks + i / 32), 4);
  uint8_t byte = w[o * (n_in / 2) + i / 2];
  int v = (i % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
  int q = (v >= 8) ? v - 16 : v;
  return scaled(d, q);
}

/* Byte size of a weight in the host layout (the WeightRef::bytes figure). */
int64_t oracle_weight_bytes(int format, int64_t n_out, int64_t n_in) {
  if (format == ORACLE_BF16) return 2 * n_out * n_in;
  if (format == ORACLE_Q8) return n_out * n_in + 4 * n_out * (n_in / 32);
  if (format == ORACLE_Q4) return n_out * (n_in / 2) + 4 * n_out * (n_in / 32);
  return -1;
}

/* Dequantise the whole weight to out[n_out][n_in] (fp32). */
int oracle_dequant(int format, const void* w, int64_t n_out, int64_t n_in, float* out) {
  if (format < 0 || format > 2) return -1;
  if (format != ORACLE_BF16 && n_in % 32 != 0) return -2;
  for (int64_t o = 0; o < n_out; ++o)
    for (int64_t i = 0; i < n_in; ++i)
      out[o * n_in + i] = weight_at(format, (const uint8_t*)w, n_out, n_in, o, i);
  return 0;
}

/* One job: y_ref[t][n_out] and mag[t][n_out] in f64 over all tokens.
 * Each weight row is dequantised once into `row` (caller scratch of n_in
 * floats); then every token's dot product runs over it with i ascending. */
int oracle_linear(int format, const void* w, int64_t n_out, int64_t n_in,
                  const float* x, int64_t t, double* y_ref, double* mag, float* row) {
  if (format < 0 || format > 2) return -1;
  if (format != ORACLE_BF16 && n_in % 32 != 0) return -2;
  for (int64_t o = 0; o < n_out; ++o) {
    for (int64_t i = 0; i < n_in; ++i)
      row[i] = weight_at(format, (const uint8_t*)w, n_out, n_in, o, i);
    for (int64_t tt = 0; tt < t; ++tt) {
      double acc = 0.0, m = 0.0;
      const float* xr = x + tt * n_in;
      for (int64_t i = 0; i < n_in; ++i) {
        double p = (double)xr[i] * (double)row[i];
        acc += p;
        m += fabs(p);
      }
      y_ref[tt * n_out + o] = acc;
      mag[tt * n_out + o] = m;
    }
  }
  return 0;
}

/* Sampled outputs: for each s, the single element (tok[s], row[s]) of one job,
 * computed straight from the definition.  Used at sizes where the full
 * product would take the CPU too long. */
int oracle_linear_sampled(int format, const void* w, int64_t n_out, int64_t n_in,
                          const float* x, int64_t t, int64_t n_samples,
                          const int64_t* tok, const int64_t* row, double* y_ref,
                          double* mag) {
  if (format < 0 || format > 2) return -1;
  if (format != ORACLE_BF16 && n_in % 32 != 0) return -2;
  for (int64_t s = 0; s < n_samples; ++s) {
    if (tok[s] < 0 || tok[s] >= t || row[s] < 0 || row[s] >= n_out) return -3;
    const float* xr = x + tok[s] * n_in;
    double acc = 0.0, m = 0.0;
    for (int64_t i = 0; i < n_in; ++i) {
      double p = (double)xr[i] *
                 (double)weight_at(format, (const uint8_t*)w, n_out, n_in, row[s], i);
      acc += p;
      m += fabs(p);
    }
    y_ref[s] = acc;
    mag[s] = m;
  }
  return 0;
}

/* gelu_mul, the step that follows the shared-input gate+up batch in the pages'
 * drafter (oxinfer 0.0.1, src/drafter.rs, `Drafter::step`: `matmul_multi` over
 * gate and up, then `gelu_mul(&mut g, &u)`).  The pages do not print gelu_mul;
 * the reading taken is g[i] <- gelu(g[i]) * u[i] with gelu in the tanh form of
 * the Gemma family the pages serve:
 *   gelu(g) = 0.5 * g * (1 + tanh(sqrt(2/pi) * (g + 0.044715 * g^3))).
 * Evaluated in double. */
double oracle_gelu(double g) {
  const double pi = acos(-1.0);
  const double inner = sqrt(2.0 / pi) * (g + 0.044715 * g * g * g);
  return 0.5 * g * (1.0 + tanh(inner));
}

/* h[i] = gelu(g[i]) * u[i] for i < n (g: gate results, u: up results). */
void oracle_gelu_mul(const double* g, const double* u, int64_t n, double* h) {
  for (int64_t i = 0; i < n; ++i) h[i] = oracle_gelu(g[i]) * u[i];
}
