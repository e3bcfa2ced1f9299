/*
 * csa2_oracle.h -- the CSA2 oracle: a plain, slow, fp64 CPU statement of what
 * the CSA2 global-attention step computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only the tests, the package smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no source with the CUDA library.
 *
 * Pages cited (the method is described only in prose on them):
 *   [P3] "Unlocking Extreme Context Scaling with DeepSeek-V4.1-Flash",
 *        sections "Compressed Sparse Attention 2 (CSA2)" and
 *        "Deployment and Infrastructure".
 *   [P4] aiany.app item page on DeepSeek-V4.1-Flash, section
 *        "What Sets It Apart".
 *   [P5] "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
 *        (Daily Paper Cast transcript), sections Introduction and Method.
 *   [MX] OCP Microscaling Formats (MX) Specification v1.0: E2M1 element
 *        encoding and the shared power-of-two (UE8M0) block scale.
 *
 * All floating-point inputs are passed as double arrays holding the exact
 * values of the bf16 / fp32 tensors (every bf16 and fp32 value is a double).
 * Every function here is single-threaded per output element; OpenMP only
 * distributes independent outputs (rows or (query, entry) pairs) across
 * threads and never changes the order of any sum.
 */
#ifndef CSA2_ORACLE_H
#define CSA2_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ---------------------------------------------------- */

/* E2M1 (4-bit: sign bit 3, two exponent bits, one mantissa bit, bias 1) [P4][MX]. */
double oracle_e2m1_value(int code);
/* UE8M0 block scale byte s -> 2^(s-127); s = 255 is never produced. [MX] */
double oracle_ue8m0_value(int s);
/* E4M3 ("fn": bias 7, no infinities, S.1111.111 is NaN), the FP8 indexer-K format. */
double oracle_e4m3_value(int b);
/* Nearest E2M1 code to y, ties to the even code, |y| > 6 saturates to 6, sign kept. */
int oracle_e2m1_encode(double y);
/* Nearest E4M3 code to x, ties to the even code, |x| > 448 saturates to 448, sign kept. */
int oracle_e4m3_encode(double x);
/* floor(log2(a)) for finite a > 0, exact (no libm log). */
int oracle_floor_log2(double a);

/* ---- a1: FP4 quantiser ------------------------------------------------- */

/* x: [rows, d] values (bf16 in the product), d % 32 == 0.
 * codes: [rows, d/2] bytes, element 2i in the low nibble of byte i.
 * scales: [rows, d/32] UE8M0 bytes.  Returns 0, or -1 on a bad argument. */
int oracle_quantize_fp4(const double* x, int64_t rows, int32_t d,
                        uint8_t* codes, uint8_t* scales);
/* Dequantise: out[r, i] = e2m1(code) * 2^(scale - 127). */
void oracle_dequantize_fp4(const uint8_t* codes, const uint8_t* scales,
                           int64_t rows, int32_t d, double* out);
/* Element-wise E4M3 cast (no scale) of the indexer-K rows. */
void oracle_cast_e4m3(const double* x, int64_t n, uint8_t* out);

/* ---- a2: indexer-Q quantiser ------------------------------------------- */

/* q: [nq, hi, di]; w: [nq, hi].  Per (row, head): sigma = 2^e with e the
 * smallest integer such that amax / sigma <= 448 (e >= -126); amax = 0 gives
 * sigma = 1 and all-zero codes.  q8 = e4m3(q / sigma); c = w * sigma. */
void oracle_quantize_index_q(const double* q, const double* w, int64_t nq,
                             int32_t hi, int32_t di, uint8_t* q8, double* c);

/* ---- a3: indexer score ------------------------------------------------- */

/* s[q, j] = sum_h c[q,h] * max(0, sum_i qv[q,h,i] * kv[b(q), j, i])  for
 * j < n_valid[q], -inf otherwise.  b(q) = q / q_per_seq.
 * qv: [nq, hi, di]; c: [nq, hi]; kv: [B, n, di]; n_valid may be NULL (= n).
 * scores: [nq, n]. */
void oracle_index_score(const double* qv, const double* c, const double* kv,
                        int64_t nq, int64_t q_per_seq, int32_t hi, int32_t di,
                        int64_t n, const int32_t* n_valid, double* scores);

/* ---- a4: top-k ---------------------------------------------------------- */

/* Per row: the min(k, n_valid) visible entries largest by (score desc,
 * index asc); written ascending by index, the rest of the row set to -1. */
void oracle_topk(const double* scores, int64_t rows, int64_t n,
                 const int32_t* n_valid, int32_t k, int32_t* idx_out);

/* ---- a5: sparse attention ---------------------------------------------- */

/* For query q of sequence b = q / q_per_seq, each head h:
 *   keys = { dequant(codes/scales of row idx[q, t]) : idx[q, t] >= 0 }
 *        U { window[b, win_start[q] + u] : 0 <= u < win_len[q] }
 *   logit_i = scale * <q_h, key_i>;  p = softmax(logit);  out = sum_i p_i key_i
 * (keys are also the values).  No key at all gives a zero output.
 * q: [nq, hq, d]; codes: [B, n, d/2]; scales: [B, n, d/32]; idx: [nq, k];
 * window: [B, w_rows, d]; win_start / win_len: [nq] or NULL (0 / w_rows).
 * out: [nq, hq, d].  Returns 0, or -1 if an index is outside [-1, n). */
int oracle_sparse_attn(const double* q, int64_t nq, int64_t q_per_seq,
                       int32_t hq, int32_t d,
                       const uint8_t* codes, const uint8_t* scales, int64_t n,
                       const int32_t* idx, int32_t k,
                       const double* window, int32_t w_rows,
                       const int32_t* win_start, const int32_t* win_len,
                       double scale, double* out);

#ifdef __cplusplus
}
#endif
#endif
