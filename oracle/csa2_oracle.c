/*
 * csa2_oracle.c -- fp64 CPU oracle for the CSA2 global-attention step.
 *
 * TEST INFRASTRUCTURE ONLY (see csa2_oracle.h).  Written to be read against
 * the definitions, not to be fast: nearest-grid searches instead of bit
 * tricks, full sorts instead of selection, one softmax per (query, head).
 *
 * Every step follows the pages' order; where they leave a step open the
 * reading taken is stated at the function.
 */
#include "csa2_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* E2M1 magnitudes by the low three code bits: exponent bits 2..1, mantissa
 * bit 0, bias 1; exponent field 0 is subnormal (0 and 0.5). [P4 "E2M1"][MX] */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_value(int code) {
  double m = E2M1_MAG[code & 7];
  return (code & 8) ? -m : m;
}

double oracle_ue8m0_value(int s) { return ldexp(1.0, s - 127); }

double oracle_e4m3_value(int b) {
  int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m / 8.0, -6); /* subnormal: 0.mmm x 2^-6 */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

int oracle_floor_log2(double a) {
  int e;
  (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
  return e - 1;
}

/* Index of the grid point nearest to a >= 0 in an ascending grid whose
 * entry i is the magnitude of code i; ties go to the even code (the code
 * whose mantissa lsb is 0); a at or above the top saturates to the top. */
static int nearest_code(const double* grid, int ngrid, double a) {
  if (a >= grid[ngrid - 1]) return ngrid - 1;
  int lo = 0, hi = ngrid - 1; /* grid[lo] <= a < grid[hi] */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (grid[mid] <= a)
      lo = mid;
    else
      hi = mid;
  }
  double dl = a - grid[lo], dh = grid[hi] - a;
  if (dl < dh) return lo;
  if (dh < dl) return hi;
  return (lo % 2 == 0) ? lo : hi;
}

int oracle_e2m1_encode(double y) {
  int neg = signbit(y) ? 1 : 0;
  int c = nearest_code(E2M1_MAG, 8, fabs(y));
  return c | (neg << 3);
}

static double E4M3_MAG[127]; /* codes 0x00 .. 0x7e; 0x7e = 448 */
static int e4m3_ready = 0;

static void e4m3_init(void) {
  if (e4m3_ready) return;
  for (int c = 0; c < 127; ++c) E4M3_MAG[c] = oracle_e4m3_value(c);
  e4m3_ready = 1;
}

int oracle_e4m3_encode(double x) {
  e4m3_init();
  if (isnan(x)) return 0x7f;
  int neg = signbit(x) ? 1 : 0;
  int c = nearest_code(E4M3_MAG, 127, fabs(x));
  return c | (neg << 7);
}

/* ------------------------------------------------------------------------ */
/* a1: FP4 quantiser                                                         */
/* ------------------------------------------------------------------------ */

/* [P4 "What Sets It Apart"] names the main-KV format E2M1 FP4; [P3
 * "Deployment and Infrastructure"] says the main KV cache is FP4-quantised.
 * The per-32-element power-of-two scale and its rule are those of [MX]:
 * X = 2^(floor(log2 amax) - 2), 2 being the largest E2M1 exponent, so
 * amax / X lies in [4, 8) and magnitudes above 6 clip to 6.
 * Readings: amax = 0 gives scale byte 0 and all-zero codes; the scale
 * exponent is clamped to [-127, 127]; zero results keep their sign. */
int oracle_quantize_fp4(const double* x, int64_t rows, int32_t d,
                        uint8_t* codes, uint8_t* scales) {
  if (d <= 0 || d % 32 != 0 || rows < 0) return -1;
  e4m3_init();
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const double* xr = x + r * d;
    uint8_t* cr = codes + r * (d / 2);
    memset(cr, 0, (size_t)(d / 2));
    for (int32_t blk = 0; blk < d / 32; ++blk) {
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) {
        double a = fabs(xr[blk * 32 + i]);
        if (a > amax) amax = a;
      }
      if (amax == 0.0) {
        scales[r * (d / 32) + blk] = 0;
        continue; /* codes stay 0 */
      }
      int e = oracle_floor_log2(amax) - 2;
      if (e < -127) e = -127;
      if (e > 127) e = 127;
      scales[r * (d / 32) + blk] = (uint8_t)(e + 127);
      for (int i = 0; i < 32; ++i) {
        int el = blk * 32 + i;
        double y = ldexp(xr[el], -e); /* exact: division by a power of two */
        int c = oracle_e2m1_encode(y);
        cr[el / 2] |= (uint8_t)((el % 2 == 0) ? c : (c << 4));
      }
    }
  }
  return 0;
}

void oracle_dequantize_fp4(const uint8_t* codes, const uint8_t* scales,
                           int64_t rows, int32_t d, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int32_t i = 0; i < d; ++i) {
      uint8_t byte = codes[r * (d / 2) + i / 2];
      int c = (i % 2 == 0) ? (byte & 15) : (byte >> 4);
      out[r * d + i] =
          oracle_e2m1_value(c) * oracle_ue8m0_value(scales[r * (d / 32) + i / 32]);
    }
}

void oracle_cast_e4m3(const double* x, int64_t n, uint8_t* out) {
  e4m3_init();
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_e4m3_encode(x[i]);
}

/* ------------------------------------------------------------------------ */
/* a2: indexer-Q quantiser                                                   */
/* ------------------------------------------------------------------------ */

/* The pages name an indexer Q and an FP8 indexer K [P3 "CSA2"] but not the
 * precision of Q.  Reading: Q is cast to E4M3 per (row, head) with the
 * smallest power-of-two scale that keeps every element within the E4M3
 * range, so the contraction is FP8 x FP8; the scale is folded into the head
 * weight (c = w * sigma), which leaves s = sum_h c_h ReLU(q8_h . k) equal in
 * exact arithmetic to the score of the scaled-back Q. */
void oracle_quantize_index_q(const double* q, const double* w, int64_t nq,
                             int32_t hi, int32_t di, uint8_t* q8, double* c) {
  e4m3_init();
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nq * hi; ++r) {
    const double* qr = q + r * di;
    double amax = 0.0;
    for (int32_t i = 0; i < di; ++i)
      if (fabs(qr[i]) > amax) amax = fabs(qr[i]);
    if (amax == 0.0) {
      memset(q8 + r * di, 0, (size_t)di);
      c[r] = w[r];
      continue;
    }
    /* smallest e with amax / 2^e <= 448, searched upward from a value that
     * is certainly too small (amax / 2^(floor(log2 amax) - 9) >= 512) */
    int e = oracle_floor_log2(amax) - 9;
    while (ldexp(amax, -e) > 448.0) ++e;
    if (e < -126) e = -126;
    for (int32_t i = 0; i < di; ++i)
      q8[r * di + i] = (uint8_t)oracle_e4m3_encode(ldexp(qr[i], -e));
    c[r] = ldexp(w[r], e);
  }
}

/* ------------------------------------------------------------------------ */
/* a3: indexer score                                                         */
/* ------------------------------------------------------------------------ */

/* The indexer scores every compressed entry visible to a query with the
 * layer's indexer Q against the indexer K [P3 "CSA2": Full mode computes
 * indexer K afresh, Reindex scores with a local indexer Q].  The formula,
 * a w-weighted sum over heads of ReLU(q_h . k_j), is the build's definition
 * (the pages give none).  Entries j >= n_valid[q] are not visible: -inf. */
void oracle_index_score(const double* qv, const double* c, const double* kv,
                        int64_t nq, int64_t q_per_seq, int32_t hi, int32_t di,
                        int64_t n, const int32_t* n_valid, double* scores) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t q = 0; q < nq; ++q)
    for (int64_t j = 0; j < n; ++j) {
      int64_t nv = n_valid ? n_valid[q] : n;
      if (j >= nv) {
        scores[q * n + j] = -INFINITY;
        continue;
      }
      const double* kj = kv + ((q / q_per_seq) * n + j) * di;
      double s = 0.0;
      for (int32_t h = 0; h < hi; ++h) {
        const double* qh = qv + (q * hi + h) * di;
        double dot = 0.0;
        for (int32_t i = 0; i < di; ++i) dot += qh[i] * kj[i];
        s += c[q * hi + h] * (dot > 0.0 ? dot : 0.0);
      }
      scores[q * n + j] = s;
    }
}

/* ------------------------------------------------------------------------ */
/* a4: top-k                                                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
  double s;
  int64_t j;
} scored_t;

/* score descending, then index ascending; +0 and -0 compare equal */
static int cmp_scored(const void* pa, const void* pb) {
  const scored_t* a = (const scored_t*)pa;
  const scored_t* b = (const scored_t*)pb;
  if (a->s > b->s) return -1;
  if (a->s < b->s) return 1;
  return (a->j < b->j) ? -1 : (a->j > b->j);
}

static int cmp_int32(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

/* Full mode selects new Top-512 entries [P3 "CSA2"].  Ties go to the lower
 * index; the chosen indices are written in ascending order and a row with
 * fewer than k visible entries is padded with -1. */
void oracle_topk(const double* scores, int64_t rows, int64_t n,
                 const int32_t* n_valid, int32_t k, int32_t* idx_out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < rows; ++r) {
    int64_t nv = n_valid ? n_valid[r] : n;
    if (nv > n) nv = n;
    if (nv < 0) nv = 0;
    scored_t* all = (scored_t*)malloc(sizeof(scored_t) * (size_t)(nv > 0 ? nv : 1));
    for (int64_t j = 0; j < nv; ++j) {
      all[j].s = scores[r * n + j];
      all[j].j = j;
    }
    qsort(all, (size_t)nv, sizeof(scored_t), cmp_scored);
    int64_t m = nv < k ? nv : k;
    int32_t* out = idx_out + r * k;
    for (int64_t t = 0; t < m; ++t) out[t] = (int32_t)all[t].j;
    qsort(out, (size_t)m, sizeof(int32_t), cmp_int32);
    for (int64_t t = m; t < k; ++t) out[t] = -1;
    free(all);
  }
}

/* ------------------------------------------------------------------------ */
/* a5: sparse attention over gathered FP4 rows joined with the SWA window     */
/* ------------------------------------------------------------------------ */

/* The selected compressed entries are gathered from the FP4 main KV cache
 * and dequantised [P4 "What Sets It Apart"; P5 Method: the inference system
 * handles the FP4 format]; the layer-local sliding window [P5 Introduction:
 * global branch beside local sliding-window attention] joins them under one
 * softmax.  Readings: one latent row is both key and value; no
 * de-duplication between the two sets; the logit scale is an argument. */
int oracle_sparse_attn(const double* q, int64_t nq, int64_t q_per_seq,
                       int32_t hq, int32_t d,
                       const uint8_t* codes, const uint8_t* scales, int64_t n,
                       const int32_t* idx, int32_t k,
                       const double* window, int32_t w_rows,
                       const int32_t* win_start, const int32_t* win_len,
                       double scale, double* out) {
  for (int64_t qi = 0; qi < nq; ++qi) {
    for (int32_t t = 0; t < k; ++t) {
      int32_t j = idx[qi * k + t];
      if (j < -1 || j >= n) return -1;
    }
    int32_t ws = win_start ? win_start[qi] : 0;
    int32_t wl = win_len ? win_len[qi] : w_rows;
    if (ws < 0 || wl < 0 || (int64_t)ws + wl > w_rows) return -1;
  }
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t qi = 0; qi < nq; ++qi) {
    int64_t b = qi / q_per_seq;
    int32_t ws = win_start ? win_start[qi] : 0;
    int32_t wl = win_len ? win_len[qi] : w_rows;
    int64_t nkeys = 0;
    double* keys = (double*)malloc(sizeof(double) * (size_t)((int64_t)(k + wl) * d + 1));
    double* logit = (double*)malloc(sizeof(double) * (size_t)(k + wl + 1));
    if (!keys || !logit) {
      bad = 1;
      free(keys);
      free(logit);
      continue;
    }
    for (int32_t t = 0; t < k; ++t) {
      int32_t j = idx[qi * k + t];
      if (j < 0) continue;
      oracle_dequantize_fp4(codes + (b * n + j) * (d / 2),
                            scales + (b * n + j) * (d / 32), 1, d,
                            keys + nkeys * d);
      ++nkeys;
    }
    for (int32_t u = 0; u < wl; ++u) {
      memcpy(keys + nkeys * d, window + (b * w_rows + ws + u) * (int64_t)d,
             sizeof(double) * (size_t)d);
      ++nkeys;
    }
    for (int32_t h = 0; h < hq; ++h) {
      const double* qh = q + (qi * hq + h) * (int64_t)d;
      double* oh = out + (qi * hq + h) * (int64_t)d;
      for (int32_t i = 0; i < d; ++i) oh[i] = 0.0;
      if (nkeys == 0) continue;
      double mx = -INFINITY;
      for (int64_t t = 0; t < nkeys; ++t) {
        double dot = 0.0;
        for (int32_t i = 0; i < d; ++i) dot += qh[i] * keys[t * d + i];
        logit[t] = scale * dot;
        if (logit[t] > mx) mx = logit[t];
      }
      double z = 0.0;
      for (int64_t t = 0; t < nkeys; ++t) {
        logit[t] = exp(logit[t] - mx);
        z += logit[t];
      }
      for (int64_t t = 0; t < nkeys; ++t) {
        double p = logit[t] / z;
        for (int32_t i = 0; i < d; ++i) oh[i] += p * keys[t * d + i];
      }
    }
    free(keys);
    free(logit);
  }
  return bad ? -2 : 0;
}
