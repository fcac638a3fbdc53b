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
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
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

/* Rows [o0, o1) of one job: y_ref[t][n_out] and mag[t][n_out] in f64 over all
 * tokens.  Each weight row is dequantised once into `row` (scratch of n_in
 * floats); then every token's dot product runs over it with i ascending. */
static void linear_rows(int format, const uint8_t* w, int64_t n_out, int64_t n_in, const float* x, int64_t t,
                        int64_t o0, int64_t o1, double* y_ref, double* mag, float* row) {
  for (int64_t o = o0; o < o1; ++o) {
    for (int64_t i = 0; i < n_in; ++i)
      row[i] = weight_at(format, w, n_out, n_in, o, i);
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
}

/* One job over all rows (caller scratch `row` of n_in floats). */
int oracle_linear(int format, const void* w, int64_t n_out, int64_t n_in,
                  const float* x, int64_t t, double* y_ref, double* mag, float* row) {
  if (format < 0 || format > 2) return -1;
  if (format != ORACLE_BF16 && n_in % 32 != 0) return -2;
  linear_rows(format, (const uint8_t*)w, n_out, n_in, x, t, 0, n_out, y_ref, mag, row);
  return 0;
}

/* The same job with its rows split into n_threads contiguous ranges, one POSIX
 * thread each.  Every element is computed exactly as by oracle_linear (same
 * dequantisation, same summation order), so the results are identical; only
 * the wall time differs.  Used to time the oracle on all host cores. */
struct rows_task {
  int format;
  const uint8_t* w;
  int64_t n_out, n_in, t, o0, o1;
  const float* x;
  double *y_ref, *mag;
  int rc;
};

static void* rows_thread(void* arg) {
  struct rows_task* k = (struct rows_task*)arg;
  float* row = (float*)malloc((size_t)k->n_in * sizeof(float));
  if (row == NULL) {
    k->rc = -4;
    return NULL;
  }
  linear_rows(k->format, k->w, k->n_out, k->n_in, k->x, k->t, k->o0, k->o1, k->y_ref, k->mag, row);
  free(row);
  k->rc = 0;
  return NULL;
}

int oracle_linear_threads(int format, const void* w, int64_t n_out, int64_t n_in, const float* x, int64_t t,
                          double* y_ref, double* mag, int n_threads) {
  if (format < 0 || format > 2) return -1;
  if (format != ORACLE_BF16 && n_in % 32 != 0) return -2;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 1024) n_threads = 1024;
  if ((int64_t)n_threads > n_out) n_threads = (int)(n_out > 0 ? n_out : 1);
  struct rows_task* tasks = (struct rows_task*)calloc((size_t)n_threads, sizeof(struct rows_task));
  pthread_t* ids = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
  int* started = (int*)calloc((size_t)n_threads, sizeof(int));
  if (tasks == NULL || ids == NULL || started == NULL) {
    free(tasks);
    free(ids);
    free(started);
    return -4;
  }
  int rc = 0;
  for (int k = 0; k < n_threads; ++k) {
    tasks[k].format = format;
    tasks[k].w = (const uint8_t*)w;
    tasks[k].n_out = n_out;
    tasks[k].n_in = n_in;
    tasks[k].t = t;
    tasks[k].o0 = n_out * k / n_threads;
    tasks[k].o1 = n_out * (k + 1) / n_threads;
    tasks[k].x = x;
    tasks[k].y_ref = y_ref;
    tasks[k].mag = mag;
    tasks[k].rc = -5;
    started[k] = pthread_create(&ids[k], NULL, rows_thread, &tasks[k]) == 0;
    if (!started[k]) rows_thread(&tasks[k]);  /* no thread: run the range here */
  }
  for (int k = 0; k < n_threads; ++k) {
    if (started[k]) pthread_join(ids[k], NULL);
    if (tasks[k].rc != 0) rc = tasks[k].rc;
  }
  free(tasks);
  free(ids);
  free(started);
  return rc;
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

/* ---------------------------------------------------------------------------
 * Centroid-masked LM head (oxinfer 0.0.1, src/drafter.rs, end of
 * `Drafter::step`): logits of the centroids, the top-k centroids, exact logits
 * over the tokens of their clusters, and the first maximum.
 *   centroids : bf16 [n_cent][h]; embed: bf16 [vocab][h]; ordering: u32 [vocab],
 *   cluster c owning ordering[c*per .. (c+1)*per), per = vocab / n_cent.
 * Readings where the page leaves the step open (the selection there is
 * `select_nth_unstable_by`, whose order and tie handling are unspecified):
 *   - the k selected centroids are the k largest logits, ties to the lower
 *     centroid index, NaN below every number; they are taken in that rank
 *     order, which is also the order the final scan visits them;
 *   - the final scan starts from (-inf, token 0) and takes a score only when it
 *     is strictly greater, so the first maximum in (rank, position) order wins,
 *     NaN and -inf never win, and with no winner the token is 0.
 * ------------------------------------------------------------------------- */

/* Rank of centroid a before centroid b: larger logit first, NaN last, ties to
 * the lower index. */
static int ranks_before(const double* cl, int64_t a, int64_t b) {
  const int na = isnan(cl[a]), nb = isnan(cl[b]);
  if (na != nb) return nb;            /* the number ranks before the NaN */
  if (!na && cl[a] != cl[b]) return cl[a] > cl[b];
  return a < b;
}

/* Step 1 and 2: centroid logits (f64) and the k selected centroids in rank order
 * (selection by repeated scans: plain and slow on purpose). */
int oracle_centroid_select(const void* centroids, int64_t n_cent, int64_t h, const float* x, int64_t k,
                           double* cl, int64_t* sel) {
  if (n_cent < 1 || h < 1 || k < 1 || k > n_cent) return -1;
  for (int64_t c = 0; c < n_cent; ++c) {
    double acc = 0.0;
    for (int64_t i = 0; i < h; ++i)
      acc += (double)x[i] * (double)weight_at(ORACLE_BF16, (const uint8_t*)centroids, n_cent, h, c, i);
    cl[c] = acc;
  }
  for (int64_t r = 0; r < k; ++r) {
    int64_t best = -1;
    for (int64_t c = 0; c < n_cent; ++c) {
      int taken = 0;
      for (int64_t q = 0; q < r; ++q) taken |= sel[q] == c;
      if (taken) continue;
      if (best < 0 || ranks_before(cl, c, best)) best = c;
    }
    sel[r] = best;
  }
  return 0;
}

/* Step 3: the exact logit of every token of the selected clusters, in
 * (rank, position) order: scores[i*per + j] = embed[ordering[sel[i]*per + j]] . x,
 * with mag = sum |embed . x| for the tolerance. */
int oracle_cluster_scores(const void* embed, int64_t vocab, int64_t h, const uint32_t* ordering, int64_t per,
                          const int64_t* sel, int64_t k, const float* x, double* scores, double* mag) {
  for (int64_t i = 0; i < k; ++i)
    for (int64_t j = 0; j < per; ++j) {
      const uint32_t tok = ordering[sel[i] * per + j];
      if ((int64_t)tok >= vocab) return -1;
      double acc = 0.0, m = 0.0;
      for (int64_t e = 0; e < h; ++e) {
        const double p = (double)x[e] * (double)weight_at(ORACLE_BF16, (const uint8_t*)embed, vocab, h, tok, e);
        acc += p;
        m += fabs(p);
      }
      scores[i * per + j] = acc;
      mag[i * per + j] = m;
    }
  return 0;
}

/* Step 4: the first maximum, strict '>' from (-inf, token 0).  Returns the
 * winning position i*per + j, or -1 when nothing beats -inf. */
int64_t oracle_first_max(const double* scores, int64_t n) {
  double best = -INFINITY;
  int64_t at = -1;
  for (int64_t p = 0; p < n; ++p)
    if (scores[p] > best) {
      best = scores[p];
      at = p;
    }
  return at;
}
