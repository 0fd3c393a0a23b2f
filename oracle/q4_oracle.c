/*
 * q4_oracle.c -- CPU oracle for the GGUF Q4_0 linear layer (TEST INFRASTRUCTURE).
 *
 * Plain C99, built with -O2 -ffp-contract=off and no fast-math, so every fp32
 * expression below is one IEEE binary32 operation in the order written.  See
 * q4_oracle.h for the format and for who may use this file.
 *
 * Method source: GeekNews on the Rust/Burn "Voxtral Mini 4B Realtime" port,
 * es.news.hada.io/topic?id=26595, section "Arquitectura" (Q4 GGUF path: GGUF
 * Q4_0 quantization, custom GPU shaders) and section "Soluciones técnicas"
 * (Q4 embedding table on the GPU with per-token row lookup).  Everything the
 * pages leave open is a stated reading, marked READING below.
 */
#define _POSIX_C_SOURCE 200809L
#include "q4_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- binary16 */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float q4o_half_to_float(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int frac = h & 0x3FF;
  float v;
  if (e == 0) {
    v = ldexpf((float)frac, -24); /* zero or subnormal: frac * 2^-24 */
  } else if (e == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexpf((float)(frac + 1024), e - 25); /* (1.frac) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* Nearest binary16 to f, ties to the even significand, overflow to +-Inf.
 * Done in double: a binary32 value and its scaled forms are exact there. */
uint16_t q4o_float_to_half_rne(float f) {
  if (isnan(f)) return 0x7E00;
  uint16_t sign = signbit(f) ? 0x8000 : 0;
  double a = fabs((double)f);
  /* 65520 = 65504 + half an ulp: from there on the nearest value is 2^16 -> Inf */
  if (a >= 65520.0) return (uint16_t)(sign | 0x7C00);
  if (a == 0.0) return sign;
  /* spacing of binary16 values around a */
  double q;
  if (a < ldexp(1.0, -14)) {
    q = ldexp(1.0, -24);
  } else {
    int e;
    frexp(a, &e); /* a = m * 2^e, m in [0.5, 1): floor(log2 a) = e - 1 */
    q = ldexp(1.0, e - 1 - 10);
  }
  double n = a / q; /* exact: division by a power of two */
  double fl = floor(n);
  double rem = n - fl;
  if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) == 1.0)) fl += 1.0;
  double v = fl * q;
  if (v == 0.0) return sign;
  if (v < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)fl); /* subnormal */
  int e2;
  frexp(v, &e2);
  int biased = (e2 - 1) + 15;
  uint16_t frac = (uint16_t)(v / ldexp(1.0, e2 - 1 - 10) - 1024.0);
  return (uint16_t)(sign | (biased << 10) | frac);
}

/* ---------------------------------------------------------------- block decode */

void q4o_decode_block(const uint8_t* blk, float* out32) {
  uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8)); /* little-endian */
  float d = q4o_half_to_float(dbits);
  for (int j = 0; j < 16; ++j) {
    int lo = blk[2 + j] & 0x0F;
    int hi = (blk[2 + j] >> 4) & 0x0F;
    out32[j] = (float)(lo - 8) * d;
    out32[j + 16] = (float)(hi - 8) * d;
  }
}

int q4o_dequant_rows(const uint8_t* blocks, int64_t n_rows, int64_t k, float* out) {
  if (!blocks || !out || n_rows < 0 || k <= 0 || k % 32) return Q4O_ERR_INVALID_ARG;
  int64_t nb = k / 32;
  for (int64_t r = 0; r < n_rows; ++r)
    for (int64_t b = 0; b < nb; ++b)
      q4o_decode_block(blocks + (r * nb + b) * 18, out + r * k + b * 32);
  return Q4O_OK;
}

/* ---------------------------------------------------------------- quantize */

/* READING (the pages give no quantizer; this is the usual GGUF Q4_0 rule, with
 * the codes taken against the stored binary16 scale):
 *   1. m = the element of largest |x|; among equal |x| the lowest index.
 *   2. d = binary16(m / -8), round to nearest even.  m == +-0 gives d = +0.
 *   3. dd = d widened to fp32.  dd == 0: every code is 8.  Otherwise each code
 *      q = clamp(floor(x / dd + 8.5), 0, 15), the division and the add each one
 *      fp32 IEEE operation.  Exact ties x/dd = n + 1/2 round up.
 *   4. byte j = q_j | (q_{j+16} << 4); d stored little-endian.
 *   A block holding NaN/Inf, or whose d rounds to +-Inf, is NONFINITE and is
 *   written as d = +0, all codes 8. */
int q4o_quantize_block(const float* x, uint8_t* blk) {
  int bad = 0;
  for (int i = 0; i < 32; ++i)
    if (!isfinite(x[i])) bad = 1;

  int im = 0;
  float amax = fabsf(x[0]);
  for (int i = 1; i < 32; ++i) {
    if (fabsf(x[i]) > amax) {
      amax = fabsf(x[i]);
      im = i;
    }
  }

  uint16_t dbits = 0;
  if (!bad && amax != 0.0f) {
    float d32 = x[im] / -8.0f;
    dbits = q4o_float_to_half_rne(d32);
    if ((dbits & 0x7C00) == 0x7C00) bad = 1; /* rounded to +-Inf */
  }
  if (bad) {
    blk[0] = 0;
    blk[1] = 0;
    memset(blk + 2, 0x88, 16);
    return Q4O_ERR_NONFINITE;
  }

  float dd = q4o_half_to_float(dbits);
  uint8_t q[32];
  for (int i = 0; i < 32; ++i) {
    if (dd == 0.0f) {
      q[i] = 8;
    } else {
      float t = x[i] / dd;
      float u = t + 8.5f;
      float fq = floorf(u);
      if (fq < 0.0f) fq = 0.0f;
      if (fq > 15.0f) fq = 15.0f;
      q[i] = (uint8_t)fq;
    }
  }
  blk[0] = (uint8_t)(dbits & 0xFF);
  blk[1] = (uint8_t)(dbits >> 8);
  for (int j = 0; j < 16; ++j) blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
  return Q4O_OK;
}

int q4o_quantize(const float* w, int64_t n, int64_t k, uint8_t* blocks, int64_t* n_bad) {
  if (!w || !blocks || n < 0 || k <= 0 || k % 32) return Q4O_ERR_INVALID_ARG;
  int64_t nb = k / 32, bad = 0;
  for (int64_t r = 0; r < n; ++r)
    for (int64_t b = 0; b < nb; ++b)
      if (q4o_quantize_block(w + r * k + b * 32, blocks + (r * nb + b) * 18) != Q4O_OK) ++bad;
  if (n_bad) *n_bad = bad;
  return bad ? Q4O_ERR_NONFINITE : Q4O_OK;
}

/* ---------------------------------------------------------------- matmul (fp64) */

typedef struct {
  const uint8_t* W;
  int64_t n, k;
  const float* X;
  int64_t m, ldx;
  double* Y;
  double* S;
  int64_t ldy;
  int64_t row_begin, row_end;
} q4o_mm_job;

static void* q4o_mm_worker(void* arg) {
  q4o_mm_job* jb = (q4o_mm_job*)arg;
  int64_t nb = jb->k / 32;
  float* wrow = (float*)malloc((size_t)jb->k * sizeof(float));
  if (!wrow) return (void*)1;
  for (int64_t i = jb->row_begin; i < jb->row_end; ++i) {
    for (int64_t b = 0; b < nb; ++b) q4o_decode_block(jb->W + (i * nb + b) * 18, wrow + b * 32);
    for (int64_t mm = 0; mm < jb->m; ++mm) {
      const float* x = jb->X + mm * jb->ldx;
      double y = 0.0, s = 0.0;
      for (int64_t kk = 0; kk < jb->k; ++kk) {
        double p = (double)wrow[kk] * (double)x[kk]; /* exact: 24x24 bits fit in 53 */
        y += p;
        s += fabs(p);
      }
      jb->Y[mm * jb->ldy + i] = y;
      if (jb->S) jb->S[mm * jb->ldy + i] = s;
    }
  }
  free(wrow);
  return NULL;
}

int q4o_matmul(const uint8_t* W, int64_t n, int64_t k, const float* X, int64_t m,
               int64_t ldx, double* Y, double* S, int64_t ldy, int nthreads) {
  if (!W || !X || !Y || n < 0 || m < 0 || k <= 0 || k % 32 || ldx < k || ldy < n)
    return Q4O_ERR_INVALID_ARG;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < nthreads) nthreads = n > 0 ? (int)n : 1;
  q4o_mm_job jobs[256];
  pthread_t tids[256];
  int started[256];
  int rc = Q4O_OK;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (q4o_mm_job){W, n, k, X, m, ldx, Y, S, ldy, n * t / nthreads, n * (t + 1) / nthreads};
    started[t] = 0;
  }
  if (nthreads == 1) {
    if (q4o_mm_worker(&jobs[0]) != NULL) rc = Q4O_ERR_INVALID_ARG;
    return rc;
  }
  for (int t = 0; t < nthreads; ++t)
    started[t] = pthread_create(&tids[t], NULL, q4o_mm_worker, &jobs[t]) == 0;
  for (int t = 0; t < nthreads; ++t) {
    if (started[t]) {
      void* ret = NULL;
      pthread_join(tids[t], &ret);
      if (ret != NULL) rc = Q4O_ERR_INVALID_ARG;
    } else if (q4o_mm_worker(&jobs[t]) != NULL) {
      rc = Q4O_ERR_INVALID_ARG;
    }
  }
  return rc;
}

/* fp64 inputs: the same sum, with x taken as given (no fp32 rounding). */
int q4o_matmul_f64(const uint8_t* W, int64_t n, int64_t k, const double* X, int64_t m,
                   int64_t ldx, double* Y, double* S, int64_t ldy, int nthreads) {
  (void)nthreads;
  if (!W || !X || !Y || n < 0 || m < 0 || k <= 0 || k % 32 || ldx < k || ldy < n)
    return Q4O_ERR_INVALID_ARG;
  int64_t nb = k / 32;
  float* wrow = (float*)malloc((size_t)k * sizeof(float));
  if (!wrow) return Q4O_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i) {
    for (int64_t b = 0; b < nb; ++b) q4o_decode_block(W + (i * nb + b) * 18, wrow + b * 32);
    for (int64_t mm = 0; mm < m; ++mm) {
      const double* x = X + mm * ldx;
      double y = 0.0, s = 0.0;
      for (int64_t kk = 0; kk < k; ++kk) {
        double p = (double)wrow[kk] * x[kk];
        y += p;
        s += fabs(p);
      }
      Y[mm * ldy + i] = y;
      if (S) S[mm * ldy + i] = s;
    }
  }
  free(wrow);
  return Q4O_OK;
}

/* ---------------------------------------------------------------- decoder glue */

/* READING (no activation on the pages): SiLU-gated unit, fp64. */
void q4o_swiglu(const double* a, const double* b, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) {
    double sig = 1.0 / (1.0 + exp(-a[i]));
    out[i] = a[i] * sig * b[i];
  }
}

/* READING: greedy decoding takes the largest logit; among equal maxima the
 * lowest index; NaN logits never win. */
int64_t q4o_argmax(const double* y, int64_t n) {
  int64_t best = -1;
  for (int64_t i = 0; i < n; ++i) {
    if (isnan(y[i])) continue;
    if (best < 0 || y[i] > y[best]) best = i;
  }
  return best;
}

/* ---------------------------------------------------------------- repacked layout */

int64_t q4o_repack_bytes(int64_t n, int64_t k) {
  if (n <= 0 || k <= 0 || k % 256) return 0;
  int64_t groups = (n + 15) / 16;
  return groups * (k / 256) * 2304;
}

/* Byte offsets, inside the repacked matrix, of element e (0..31) of block kb
 * of row r: its binary16 scale (2 bytes) and the byte holding its code, with
 * *high = 1 when the code is that byte's high nibble.  The layout is the one
 * q4.h defines: tile (r / 16, kb / 8) of 2304 bytes; rows 16G + g and
 * 16G + g + 8 (g = 0..7) pair up; a tile's column c = 16s + i (s = 0..15) sits
 * with lane L = 4g + (i % 8) / 2 of step s, as nibble
 * m = hr + 2 (i / 8) + 4 (i % 2) of that lane's step word (hr = 1 for the row
 * g + 8). */
static void q4o_tile_offsets(int64_t r, int64_t kb, int64_t e, int64_t k, int64_t* scale_off,
                             int64_t* code_off, int* high) {
  int64_t tile = ((r / 16) * (k / 256) + kb / 8) * 2304;
  int64_t rr = r % 16, g = rr % 8, hr = rr / 8, b = kb % 8;
  int64_t s = 2 * b + e / 16, i = e % 16;
  int64_t lane = 4 * g + (i % 8) / 2;
  int64_t m = hr + 2 * (i / 8) + 4 * (i % 2);
  *scale_off = tile + 32 * g + 4 * b + 2 * hr;
  *code_off = tile + 256 + 512 * (s / 4) + 16 * lane + 4 * (s % 4) + m / 2;
  *high = (int)(m % 2);
}

static void q4o_put_nibble(uint8_t* byte, int high, int q) {
  if (high) *byte = (uint8_t)((*byte & 0x0F) | (q << 4));
  else *byte = (uint8_t)((*byte & 0xF0) | q);
}

int q4o_repack(const uint8_t* W, int64_t n, int64_t k, uint8_t* R) {
  if (!W || !R || n <= 0 || k <= 0 || k % 256) return Q4O_ERR_INVALID_ARG;
  int64_t nb = k / 32, groups = (n + 15) / 16;
  for (int64_t r = 0; r < groups * 16; ++r) {
    for (int64_t kb = 0; kb < nb; ++kb) {
      const uint8_t* blk = r < n ? W + (r * nb + kb) * 18 : NULL;
      for (int e = 0; e < 32; ++e) {
        int64_t so, co;
        int high;
        q4o_tile_offsets(r, kb, e, k, &so, &co, &high);
        /* padding rows past n: d = +0 and every code 8 */
        int q = 8;
        if (blk) q = e < 16 ? (blk[2 + e] & 0x0F) : (blk[2 + e - 16] >> 4);
        q4o_put_nibble(R + co, high, q);
        if (e == 0) {
          R[so] = blk ? blk[0] : 0;
          R[so + 1] = blk ? blk[1] : 0;
        }
      }
    }
  }
  return Q4O_OK;
}

int q4o_unrepack(const uint8_t* R, int64_t n, int64_t k, uint8_t* W) {
  if (!W || !R || n <= 0 || k <= 0 || k % 256) return Q4O_ERR_INVALID_ARG;
  int64_t nb = k / 32;
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t kb = 0; kb < nb; ++kb) {
      uint8_t* blk = W + (r * nb + kb) * 18;
      for (int e = 0; e < 32; ++e) {
        int64_t so, co;
        int high;
        q4o_tile_offsets(r, kb, e, k, &so, &co, &high);
        int q = high ? (R[co] >> 4) : (R[co] & 0x0F);
        if (e == 0) {
          blk[0] = R[so];
          blk[1] = R[so + 1];
        }
        q4o_put_nibble(blk + 2 + (e % 16), e >= 16, q);
      }
    }
  }
  return Q4O_OK;
}

/* ---------------------------------------------------------------- Q4 x Q8 */

/* READING: the pages name only GGUF Q4_0 ("Arquitectura"); the integer path is
 * the usual companion of that format, and its details are this library's
 * choice.  x is quantized per 32-element block to int8 with an fp32 scale:
 * amax = max |x_j|, d = amax / 127 (fp32 IEEE division), q_j = x_j / d (fp32
 * IEEE division) rounded to the nearest integer with halves away from zero,
 * clamped to [-127, 127].  amax == 0 gives d = +0 and every q_j = 0; a block
 * holding a NaN or an infinity gives d = NaN and every q_j = 0. */
int q4o_quantize_q8(const float* x, int64_t k, int8_t* q, float* d) {
  if (!x || !q || !d || k <= 0 || k % 32) return Q4O_ERR_INVALID_ARG;
  for (int64_t b = 0; b < k / 32; ++b) {
    const float* xb = x + 32 * b;
    float amax = 0.0f;
    int finite = 1;
    for (int j = 0; j < 32; ++j) {
      if (!isfinite(xb[j])) finite = 0;
      float a = fabsf(xb[j]);
      if (a > amax) amax = a;
    }
    if (!finite) {
      d[b] = NAN;
      for (int j = 0; j < 32; ++j) q[32 * b + j] = 0;
      continue;
    }
    float db = amax / 127.0f;
    d[b] = db;
    for (int j = 0; j < 32; ++j) {
      float c = 0.0f;
      if (db != 0.0f) {
        float t = xb[j] / db;
        c = roundf(t); /* halves away from zero */
        if (c > 127.0f) c = 127.0f;
        if (c < -127.0f) c = -127.0f;
      }
      q[32 * b + j] = (int8_t)c;
    }
  }
  return Q4O_OK;
}

/* The Q4 x Q8 product of every row of X (each quantized as above) with W:
 *   y_r = sum_b d_w[r,b] * d_x[b] * sum_{j in b} (q_w[r,j] - 8) * q_x[j]
 * with the integer sums exact and the rest in fp64; S_r = sum_b of the
 * magnitudes of those block terms. */
int q4o_matmul_q8(const uint8_t* W, int64_t n, int64_t k, const float* X, int64_t m,
                  int64_t ldx, double* Y, double* S, int64_t ldy) {
  if (!W || !X || !Y || n < 0 || m < 0 || k <= 0 || k % 32 || ldx < k || ldy < n)
    return Q4O_ERR_INVALID_ARG;
  int64_t nb = k / 32;
  int8_t* q = (int8_t*)malloc((size_t)k);
  float* dx = (float*)malloc((size_t)nb * sizeof(float));
  if (!q || !dx) {
    free(q);
    free(dx);
    return Q4O_ERR_INVALID_ARG;
  }
  for (int64_t mm = 0; mm < m; ++mm) {
    q4o_quantize_q8(X + mm * ldx, k, q, dx);
    for (int64_t i = 0; i < n; ++i) {
      double y = 0.0, s = 0.0;
      for (int64_t b = 0; b < nb; ++b) {
        const uint8_t* blk = W + (i * nb + b) * 18;
        double dw = (double)q4o_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
        int64_t isum = 0;
        for (int j = 0; j < 16; ++j) {
          int lo = blk[2 + j] & 0x0F, hi = blk[2 + j] >> 4;
          isum += (int64_t)(lo - 8) * q[32 * b + j];
          isum += (int64_t)(hi - 8) * q[32 * b + j + 16];
        }
        double t = dw * (double)dx[b] * (double)isum;
        y += t;
        s += fabs(t);
      }
      Y[mm * ldy + i] = y;
      if (S) S[mm * ldy + i] = s;
    }
  }
  free(q);
  free(dx);
  return Q4O_OK;
}

/* ---------------------------------------------------------------- gather */

/* READING: the pages look rows up on the CPU; the lookup itself is "row id ->
 * decoded row".  An id outside the table yields +0.0 and an error status. */
int q4o_embed_gather(const uint8_t* table, int64_t vocab, int64_t k, const int32_t* ids,
                     int64_t n_ids, float* out) {
  if (!table || !ids || !out || vocab <= 0 || n_ids < 0 || k <= 0 || k % 32)
    return Q4O_ERR_INVALID_ARG;
  int64_t nb = k / 32;
  int rc = Q4O_OK;
  for (int64_t b = 0; b < n_ids; ++b) {
    int64_t id = ids[b];
    float* row = out + b * k;
    if (id < 0 || id >= vocab) {
      for (int64_t kk = 0; kk < k; ++kk) row[kk] = 0.0f;
      rc = Q4O_ERR_ID_OUT_OF_RANGE;
      continue;
    }
    for (int64_t j = 0; j < nb; ++j) q4o_decode_block(table + (id * nb + j) * 18, row + j * 32);
  }
  return rc;
}
