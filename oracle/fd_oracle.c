/*
 * fd_oracle.c -- fp64 CPU oracle for single-token decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent check that the CUDA
 * path is measured against.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark load it.  It shares no code, header, table or helper with
 * the CUDA library, and the CUDA library never calls it.
 *
 * What it computes is the plain, UNSPLIT definition of decode attention.  The
 * split-KV method (Flash-Decoding) reaches exactly this result up to rounding
 * order; the pages demonstrate that equality on their worked example.  So the
 * oracle is that definition written out, with no blocking, no online rescaling
 * and no split/merge:
 *
 *   for every batch row b and query head h, with kv head g = floor(h / G),
 *   G = Hq / Hkv (consecutive grouping of query heads onto KV heads):
 *     s_t = (sum_j q[b,h,j] * k[b,g,t,j]) / sqrt(d)          t in [0, L_b)
 *     m   = max_t s_t                                         (safe-softmax shift)
 *     p_t = exp(s_t - m),  l = sum_t p_t
 *     o[b,h,:] = sum_t p_t * v[b,g,t,:] / l
 *     lse[b,h] = m + ln(l)                                    (natural log)
 *   and for L_b = 0: o = 0, lse = -infinity.
 *
 * Sources (web pages; section names as printed there):
 *   - "AI Infra: math and infra optimisation in large models" (gitcode.csdn.net),
 *     section 2.3 "Safe Softmax (-M)": subtract the maximum before exponentiating;
 *     section 2.4 "why divide by sqrt(d_k)": the score scale;
 *     section 2.6, "LSE and online softmax": LSE = m + log(l);
 *     section 2.5: a decode query (length 1) needs no causal mask, all cached keys
 *     are in the past -- so only keys t < L_b take part.
 *   - "2kiu.com/news/6053916", section "weight block results with log-sum-exp":
 *     the function that returns (weighted average, m + log z) over one whole block;
 *     applied to the whole sequence it is this oracle.
 *   - "FlashDecoding interview notes" (gtnt.cn/news/53829), section three: LSE in
 *     natural log, m_i + log(l_i).
 *
 * Storage: inputs are read in their stored precision (fp32, or bf16 given as raw
 * uint16 bit patterns) and up-converted exactly to double; every product and sum
 * is then done in double.
 *
 * KV layouts:
 *   contiguous: k[b][g][t][j], shape [B, Hkv, L_cap, d]   (block_table == NULL)
 *   paged:      k[page][g][slot][j], shape [num_pages, Hkv, page_size, d]; logical
 *               token t of row b lives on page block_table[b * max_pages + t / page_size]
 *               in slot t % page_size.  Logical order is the block table's order,
 *               never the physical page number.
 *
 * Threads: OpenMP over (b, h) rows; libgomp keeps its worker pool between calls,
 * so repeated calls do not measure thread creation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { FDO_F32 = 0, FDO_BF16 = 1 };

/* Exact widening of one stored element to double. */
static double fdo_load(const void* base, int dtype, int64_t idx) {
  if (dtype == FDO_F32) {
    return (double)((const float*)base)[idx];
  }
  /* bf16 is the upper half of an IEEE binary32: shift the bits into place. */
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Offset (in elements) of element j of logical token t of kv head g, row b. */
static int64_t fdo_kv_offset(int b, int g, int64_t t, int j, int Hkv, int d, int64_t L_cap,
                             const int32_t* block_table, int max_pages, int page_size) {
  if (block_table == NULL) {
    return (((int64_t)b * Hkv + g) * L_cap + t) * d + j;
  }
  int64_t page = block_table[(int64_t)b * max_pages + t / page_size];
  int64_t slot = t % page_size;
  return ((page * Hkv + g) * page_size + slot) * d + j;
}

/*
 * fd_oracle_decode: returns 0 on success, a negative code on invalid arguments
 *   -1 bad sizes, -2 Hq not a multiple of Hkv, -3 bad dtype, -4 a seq_len outside
 *   [0, L_cap], -5 a block-table entry outside [0, num_pages), -6 out of memory.
 *
 *   q       [B, Hq, d]           stored dtype
 *   k, v    see layouts above    stored dtype
 *   L_cap   contiguous: the cache capacity per row; paged: max_pages * page_size
 *   rows    optional list of n_rows flat row ids (b * Hq + h) to compute; NULL = all.
 *           Only the listed rows of out/lse are written.
 *   out     [B, Hq, d] double, lse [B, Hq] double (natural log)
 */
int fd_oracle_decode(int B, int Hq, int Hkv, int d, int dtype,
                     const void* q, const void* k, const void* v,
                     const int32_t* seq_lens, int64_t L_cap,
                     const int32_t* block_table, int max_pages, int page_size, int64_t num_pages,
                     const int64_t* rows, int64_t n_rows,
                     double* out, double* lse, int num_threads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || L_cap < 0) return -1;
  if (Hq % Hkv != 0) return -2;
  if (dtype != FDO_F32 && dtype != FDO_BF16) return -3;
  if (block_table != NULL && (page_size <= 0 || max_pages <= 0)) return -1;
  const int G = Hq / Hkv;
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0 || seq_lens[b] > L_cap) return -4;
    if (block_table != NULL) {
      int64_t used = ((int64_t)seq_lens[b] + page_size - 1) / page_size;
      for (int64_t i = 0; i < used; ++i) {
        int32_t p = block_table[(int64_t)b * max_pages + i];
        if (p < 0 || p >= num_pages) return -5;
      }
    }
  }
  const int64_t total = rows ? n_rows : (int64_t)B * Hq;
  const double scale = 1.0 / sqrt((double)d);
  int failed = 0;

#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
  for (int64_t r = 0; r < total; ++r) {
    const int64_t row = rows ? rows[r] : r;
    const int b = (int)(row / Hq);
    const int h = (int)(row % Hq);
    const int g = h / G;
    const int64_t L = seq_lens[b];
    double* o = out + row * d;

    if (L == 0) {
      for (int j = 0; j < d; ++j) o[j] = 0.0;
      lse[row] = -INFINITY;
      continue;
    }
    double* s = (double*)malloc((size_t)L * sizeof(double));
    if (s == NULL) {
      failed |= 1;
      continue;
    }
    /* Pass 1: scaled scores. */
    for (int64_t t = 0; t < L; ++t) {
      double dot = 0.0;
      for (int j = 0; j < d; ++j) {
        double qj = fdo_load(q, dtype, row * d + j);
        double kj = fdo_load(k, dtype, fdo_kv_offset(b, g, t, j, Hkv, d, L_cap, block_table,
                                                     max_pages, page_size));
        dot += qj * kj;
      }
      s[t] = dot * scale;
    }
    /* Pass 2: the maximum (safe-softmax shift). */
    double m = s[0];
    for (int64_t t = 1; t < L; ++t) {
      if (s[t] > m) m = s[t];
    }
    /* Pass 3: shifted exponentials, their sum, and the weighted sum of values. */
    double l = 0.0;
    for (int j = 0; j < d; ++j) o[j] = 0.0;
    for (int64_t t = 0; t < L; ++t) {
      double p = exp(s[t] - m);
      l += p;
      for (int j = 0; j < d; ++j) {
        o[j] += p * fdo_load(v, dtype, fdo_kv_offset(b, g, t, j, Hkv, d, L_cap, block_table,
                                                     max_pages, page_size));
      }
    }
    for (int j = 0; j < d; ++j) o[j] /= l;
    lse[row] = m + log(l);
    free(s);
  }
  return failed ? -6 : 0;
}

/*
 * fd_oracle_decode_causal: decode with Q query tokens per row (multi-token decode, as in
 * speculative verification).  The Q tokens are the last Q positions of row b and their
 * keys and values are already in the cache, so query j (0-based) sits at position
 * L_b - Q + j and, with the causal mask of "AI Infra: math and infra optimisation in
 * large models" section 2.5 (a token sees only itself and the past), attends to the
 * keys t < L_b - Q + 1 + j.  A query that sees no key gets o = 0, lse = -infinity.
 * Everything else is fd_oracle_decode's plain definition, in fp64.
 *
 *   q  [B, Q, Hq, d]   out [B, Q, Hq, d] double   lse [B, Q, Hq] double
 *   rows: optional flat ids ((b * Q + j) * Hq + h) to compute; NULL = all.
 * Returns 0, or the error codes of fd_oracle_decode.
 */
int fd_oracle_decode_causal(int B, int Q, int Hq, int Hkv, int d, int dtype,
                            const void* q, const void* k, const void* v,
                            const int32_t* seq_lens, int64_t L_cap,
                            const int32_t* block_table, int max_pages, int page_size,
                            int64_t num_pages, const int64_t* rows, int64_t n_rows,
                            double* out, double* lse, int num_threads) {
  if (B < 0 || Q <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || L_cap < 0) return -1;
  if (Hq % Hkv != 0) return -2;
  if (dtype != FDO_F32 && dtype != FDO_BF16) return -3;
  if (block_table != NULL && (page_size <= 0 || max_pages <= 0)) return -1;
  const int G = Hq / Hkv;
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0 || seq_lens[b] > L_cap) return -4;
    if (block_table != NULL) {
      int64_t used = ((int64_t)seq_lens[b] + page_size - 1) / page_size;
      for (int64_t i = 0; i < used; ++i) {
        int32_t p = block_table[(int64_t)b * max_pages + i];
        if (p < 0 || p >= num_pages) return -5;
      }
    }
  }
  const int64_t total = rows ? n_rows : (int64_t)B * Q * Hq;
  const double scale = 1.0 / sqrt((double)d);
  int failed = 0;

#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
  for (int64_t r = 0; r < total; ++r) {
    const int64_t row = rows ? rows[r] : r;          /* (b * Q + j) * Hq + h */
    const int h = (int)(row % Hq);
    const int j = (int)((row / Hq) % Q);
    const int b = (int)(row / ((int64_t)Hq * Q));
    const int g = h / G;
    const int64_t visible = (int64_t)seq_lens[b] - Q + 1 + j;   /* keys t < visible */
    double* o = out + row * d;
    if (visible <= 0) {
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      lse[row] = -INFINITY;
      continue;
    }
    double* s = (double*)malloc((size_t)visible * sizeof(double));
    if (s == NULL) {
      failed |= 1;
      continue;
    }
    for (int64_t t = 0; t < visible; ++t) {
      double dot = 0.0;
      for (int c = 0; c < d; ++c) {
        double qc = fdo_load(q, dtype, row * d + c);
        double kc = fdo_load(k, dtype, fdo_kv_offset(b, g, t, c, Hkv, d, L_cap, block_table,
                                                     max_pages, page_size));
        dot += qc * kc;
      }
      s[t] = dot * scale;
    }
    double m = s[0];
    for (int64_t t = 1; t < visible; ++t) {
      if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t t = 0; t < visible; ++t) {
      double p = exp(s[t] - m);
      l += p;
      for (int c = 0; c < d; ++c) {
        o[c] += p * fdo_load(v, dtype, fdo_kv_offset(b, g, t, c, Hkv, d, L_cap, block_table,
                                                     max_pages, page_size));
      }
    }
    for (int c = 0; c < d; ++c) o[c] /= l;
    lse[row] = m + log(l);
    free(s);
  }
  return failed ? -6 : 0;
}

/*
 * FP8 E4M3 code -> double, from the format's definition: 1 sign bit, 4 exponent bits
 * (bias 7), 3 mantissa bits; exponent 0 is subnormal (2^-6 * m / 8); the code with all
 * exponent and mantissa bits set is NaN; there is no infinity.
 */
double fd_oracle_e4m3_to_double(uint8_t code) {
  const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) {
    mag = ldexp((double)m / 8.0, -6);
  } else {
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  }
  return sign ? -mag : mag;
}

/*
 * fd_oracle_decode_kv8: single-token decode over a KV cache stored as FP8 E4M3 codes
 * with one dequantisation scale per kv head for K and for V: k = code * k_scale[g],
 * v = code * v_scale[g], widened exactly to double.  q is fp32 or bf16 (q_dtype).  The
 * attention itself is fd_oracle_decode's plain unsplit definition.
 *   q [B, Hq, d]; k, v as uint8 codes in fd_oracle_decode's layouts; out [B, Hq, d]
 *   double; lse [B, Hq] double.  Returns 0 or fd_oracle_decode's error codes.
 */
int fd_oracle_decode_kv8(int B, int Hq, int Hkv, int d, int q_dtype, const void* q,
                         const uint8_t* k, const uint8_t* v, const float* k_scale,
                         const float* v_scale, const int32_t* seq_lens, int64_t L_cap,
                         const int32_t* block_table, int max_pages, int page_size,
                         int64_t num_pages, const int64_t* rows, int64_t n_rows,
                         double* out, double* lse, int num_threads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || L_cap < 0) return -1;
  if (Hq % Hkv != 0) return -2;
  if (q_dtype != FDO_F32 && q_dtype != FDO_BF16) return -3;
  if (block_table != NULL && (page_size <= 0 || max_pages <= 0)) return -1;
  const int G = Hq / Hkv;
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0 || seq_lens[b] > L_cap) return -4;
    if (block_table != NULL) {
      int64_t used = ((int64_t)seq_lens[b] + page_size - 1) / page_size;
      for (int64_t i = 0; i < used; ++i) {
        int32_t p = block_table[(int64_t)b * max_pages + i];
        if (p < 0 || p >= num_pages) return -5;
      }
    }
  }
  const int64_t total = rows ? n_rows : (int64_t)B * Hq;
  const double scale = 1.0 / sqrt((double)d);
  int failed = 0;

#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
  for (int64_t r = 0; r < total; ++r) {
    const int64_t row = rows ? rows[r] : r;
    const int b = (int)(row / Hq);
    const int h = (int)(row % Hq);
    const int g = h / G;
    const int64_t L = seq_lens[b];
    const double ks = (double)k_scale[g], vs = (double)v_scale[g];
    double* o = out + row * d;
    if (L == 0) {
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      lse[row] = -INFINITY;
      continue;
    }
    double* s = (double*)malloc((size_t)L * sizeof(double));
    if (s == NULL) {
      failed |= 1;
      continue;
    }
    for (int64_t t = 0; t < L; ++t) {
      double dot = 0.0;
      for (int c = 0; c < d; ++c) {
        const double kc = fd_oracle_e4m3_to_double(
            k[fdo_kv_offset(b, g, t, c, Hkv, d, L_cap, block_table, max_pages, page_size)]);
        dot += fdo_load(q, q_dtype, row * d + c) * (kc * ks);
      }
      s[t] = dot * scale;
    }
    double m = s[0];
    for (int64_t t = 1; t < L; ++t) {
      if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t t = 0; t < L; ++t) {
      const double p = exp(s[t] - m);
      l += p;
      for (int c = 0; c < d; ++c) {
        const double vc = fd_oracle_e4m3_to_double(
            v[fdo_kv_offset(b, g, t, c, Hkv, d, L_cap, block_table, max_pages, page_size)]);
        o[c] += p * (vc * vs);
      }
    }
    for (int c = 0; c < d; ++c) o[c] /= l;
    lse[row] = m + log(l);
    free(s);
  }
  return failed ? -6 : 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int fd_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
