/*
 * FP64 CPU oracle of the quantized weight-streaming GEMV (definitions and
 * citations in oracle.h).
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the CPU
 * baseline of the benchmark, never by the product library.
 *
 * Plain loops, no blocking, no SIMD, no fused multiply-add (built with
 * -ffp-contract=off).  Row loops may run on several threads; each output
 * depends on its own row only, so the results do not depend on the thread
 * count.
 */
#include "oracle.h"

#include <math.h>
#include <stddef.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads for the row loops from now on (n >= 1); the timing harness uses it
 * to time the same code on one core. */
void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* binary16, from the IEEE 754 definition: 1 sign bit, 5 exponent bits (bias  */
/* 15), 10 fraction bits; subnormals are f * 2^-24.                           */
/* ------------------------------------------------------------------------ */

static const double TWO_M24 = 5.9604644775390625e-08; /* 2^-24, the subnormal step   */
static const double TWO_M14 = 6.103515625e-05;        /* 2^-14, the smallest normal  */

float orc_float_from_half(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int f = h & 1023;
  double v;
  if (e == 0) {
    v = (double)f * TWO_M24;
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25);
  }
  return (float)(sign ? -v : v);
}

uint16_t orc_half_from_float(float x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs((double)x);
  if (isnan(x)) return (uint16_t)(sign | 0x7E00);
  if (isinf(x)) return (uint16_t)(sign | 0x7C00);
  /* The spacing of binary16 values around a: 2^-24 below 2^-14, else
   * 2^(floor(log2 a) - 10).  a / spacing is exact (power-of-two scaling), and
   * rint() in the default rounding mode rounds it to nearest, ties to even. */
  double step;
  if (a < TWO_M14) {
    step = TWO_M24;
  } else {
    int ex;
    (void)frexp(a, &ex); /* a = m * 2^ex, m in [0.5, 1) */
    step = ldexp(1.0, ex - 1 - 10);
  }
  double v = rint(a / step) * step; /* nearest binary16 magnitude (may be 2^16) */
  if (v >= 65536.0) return (uint16_t)(sign | 0x7C00); /* beyond 65504 rounds to infinity */
  if (v < TWO_M14) return (uint16_t)(sign | (uint16_t)(v / TWO_M24));
  int ex;
  double m = frexp(v, &ex); /* v = (2m) * 2^(ex-1), 2m in [1, 2) */
  int e = ex - 1 + 15;
  uint16_t frac = (uint16_t)((2.0 * m - 1.0) * 1024.0);
  return (uint16_t)(sign | (uint16_t)(e << 10) | frac);
}

/* ------------------------------------------------------------------------ */
/* Q8_0                                                                       */
/* ------------------------------------------------------------------------ */

#define Q8_0_QK 32
#define Q8_0_BYTES 34
#define PQ2_0_QK 128
#define PQ2_0_BYTES 34
#define PTQ1_0_QK 128
#define SCALE4_QK 32
#define SCALE4_BYTES 18 /* fp16 scale, then 16 bytes of nibbles */
#define PTQ1_0_BYTES 28 /* 24 bytes of five trits, 2 of four trits, then the fp16 scale */

int orc_q8_0_quantize(const float* w, int64_t n, int64_t k, uint8_t* blocks) {
  if (n < 0 || k <= 0 || k % Q8_0_QK != 0) return ORC_ERR_SHAPE;
  int64_t nb = k / Q8_0_QK;
  for (int64_t i = 0; i < n * k; ++i)
    if (!isfinite(w[i])) return ORC_ERR_NONFINITE;
  int status = ORC_OK;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* wb = w + r * k + b * Q8_0_QK;
      uint8_t* out = blocks + (r * nb + b) * Q8_0_BYTES;
      float amax = 0.0f;
      for (int j = 0; j < Q8_0_QK; ++j) {
        float a = fabsf(wb[j]);
        if (a > amax) amax = a;
      }
      float d = amax / 127.0f; /* fp32 quotient */
      uint16_t dh = orc_half_from_float(d);
      if ((dh & 0x7C00) == 0x7C00) {
#pragma omp atomic write
        status = ORC_ERR_RANGE;
      }
      float df = orc_float_from_half(dh);
      out[0] = (uint8_t)(dh & 0xFF);
      out[1] = (uint8_t)(dh >> 8);
      for (int j = 0; j < Q8_0_QK; ++j) {
        long q = 0;
        if (df != 0.0f) {
          q = lround((double)wb[j] / (double)df); /* half away from zero */
          if (q > 127) q = 127;
          if (q < -127) q = -127;
        }
        out[2 + j] = (uint8_t)(int8_t)q;
      }
    }
  }
  return status;
}

int orc_q8_0_dequant(const uint8_t* blocks, int64_t n, int64_t k, float* w_out) {
  if (n < 0 || k <= 0 || k % Q8_0_QK != 0) return ORC_ERR_SHAPE;
  int64_t nb = k / Q8_0_QK;
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (r * nb + b) * Q8_0_BYTES;
      float d = orc_float_from_half((uint16_t)(blk[0] | (blk[1] << 8)));
      for (int j = 0; j < Q8_0_QK; ++j) {
        int q = (int8_t)blk[2 + j];
        w_out[r * k + b * Q8_0_QK + j] = (float)q * d; /* exact: 8-bit times 11-bit significand */
      }
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* PQ2_0                                                                      */
/* ------------------------------------------------------------------------ */

int orc_pq2_0_quantize(const float* w_rot, int64_t n, int64_t k, uint8_t* blocks) {
  if (n < 0 || k <= 0 || k % PQ2_0_QK != 0) return ORC_ERR_SHAPE;
  int64_t nb = k / PQ2_0_QK;
  for (int64_t i = 0; i < n * k; ++i)
    if (!isfinite(w_rot[i])) return ORC_ERR_NONFINITE;
  int status = ORC_OK;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* wb = w_rot + r * k + b * PQ2_0_QK;
      uint8_t* out = blocks + (r * nb + b) * PQ2_0_BYTES;
      float amax = 0.0f;
      for (int j = 0; j < PQ2_0_QK; ++j) {
        float a = fabsf(wb[j]);
        if (a > amax) amax = a;
      }
      uint16_t dh = orc_half_from_float(amax); /* d = max|w| over the group */
      if ((dh & 0x7C00) == 0x7C00) {
#pragma omp atomic write
        status = ORC_ERR_RANGE;
      }
      float df = orc_float_from_half(dh);
      memset(out, 0, PQ2_0_BYTES);
      out[0] = (uint8_t)(dh & 0xFF);
      out[1] = (uint8_t)(dh >> 8);
      for (int j = 0; j < PQ2_0_QK; ++j) {
        long t = 0;
        if (df != 0.0f) {
          t = lround((double)wb[j] / (double)df);
          if (t > 1) t = 1;
          if (t < -1) t = -1;
        }
        unsigned code = (unsigned)(t + 1); /* 0, 1 or 2 */
        out[2 + j / 4] |= (uint8_t)(code << (2 * (j % 4)));
      }
    }
  }
  return status;
}

int orc_pq2_0_dequant(const uint8_t* blocks, int64_t n, int64_t k, float* w_out) {
  if (n < 0 || k <= 0 || k % PQ2_0_QK != 0) return ORC_ERR_SHAPE;
  int64_t nb = k / PQ2_0_QK;
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (r * nb + b) * PQ2_0_BYTES;
      float d = orc_float_from_half((uint16_t)(blk[0] | (blk[1] << 8)));
      for (int j = 0; j < PQ2_0_QK; ++j) {
        int code = (blk[2 + j / 4] >> (2 * (j % 4))) & 3;
        w_out[r * k + b * PQ2_0_QK + j] = (float)(code - 1) * d;
      }
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* PTQ1_0: the same trits and scale as PQ2_0, packed in base 3                 */
/* ------------------------------------------------------------------------ */

/* Byte and trit index of element e of a block (the page's element-order
 * table): 0-79 are trit e/16 of byte e%16, 80-119 trit (e-80)/8 of byte
 * 16 + (e-80)%8, 120-127 trit (e-120)/2 of byte 24 + (e-120)%2 (qh). */
static void ptq1_0_place(int e, int* byte, int* n) {
  if (e < 80) {
    *n = e / 16;
    *byte = e % 16;
  } else if (e < 120) {
    *n = (e - 80) / 8;
    *byte = 16 + (e - 80) % 8;
  } else {
    *n = (e - 120) / 2;
    *byte = 24 + (e - 120) % 2;
  }
}

/* q = ceil(256 v / 243), v the five trits read as a base-3 number with the
 * first trit most significant (a qh byte's missing fifth trit is 0). */
static uint8_t ptq1_0_byte(const int t[5]) {
  int v = t[0] * 81 + t[1] * 27 + t[2] * 9 + t[3] * 3 + t[4];
  return (uint8_t)((256 * v + 242) / 243);
}

/* trit n of byte q: ((q * 3^n) mod 256) * 3 / 256, rounded down. */
static int ptq1_0_trit(uint8_t q, int n) {
  int p = 1;
  for (int i = 0; i < n; ++i) p *= 3;
  return ((((int)q * p) & 0xFF) * 3) >> 8;
}

int orc_ptq1_0_encode_byte(const int32_t* trits) {
  int t[5];
  for (int i = 0; i < 5; ++i) t[i] = trits[i];
  return ptq1_0_byte(t);
}

int orc_ptq1_0_decode_trit(int32_t q, int32_t n) { return ptq1_0_trit((uint8_t)q, n); }

int orc_ptq1_0_quantize(const float* w_rot, int64_t n, int64_t k, uint8_t* blocks) {
  if (n < 0 || k <= 0 || k % PTQ1_0_QK != 0) return ORC_ERR_SHAPE;
  int64_t nb = k / PTQ1_0_QK;
  for (int64_t i = 0; i < n * k; ++i)
    if (!isfinite(w_rot[i])) return ORC_ERR_NONFINITE;
  int status = ORC_OK;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* wb = w_rot + r * k + b * PTQ1_0_QK;
      uint8_t* out = blocks + (r * nb + b) * PTQ1_0_BYTES;
      float amax = 0.0f;
      for (int j = 0; j < PTQ1_0_QK; ++j) {
        float a = fabsf(wb[j]);
        if (a > amax) amax = a;
      }
      uint16_t dh = orc_half_from_float(amax); /* the PQ2_0 scale: d = max|w| over the group */
      if ((dh & 0x7C00) == 0x7C00) {
#pragma omp atomic write
        status = ORC_ERR_RANGE;
      }
      float df = orc_float_from_half(dh);
      int trits[26][5];
      memset(trits, 0, sizeof(trits));
      for (int j = 0; j < PTQ1_0_QK; ++j) {
        long t = 0;
        if (df != 0.0f) {
          t = lround((double)wb[j] / (double)df);
          if (t > 1) t = 1;
          if (t < -1) t = -1;
        }
        int byte, tn;
        ptq1_0_place(j, &byte, &tn);
        trits[byte][tn] = (int)(t + 1);
      }
      for (int byte = 0; byte < 26; ++byte) out[byte] = ptq1_0_byte(trits[byte]);
      out[26] = (uint8_t)(dh & 0xFF); /* the scale comes last */
      out[27] = (uint8_t)(dh >> 8);
    }
  }
  return status;
}

int orc_ptq1_0_dequant(const uint8_t* blocks, int64_t n, int64_t k, float* w_out) {
  if (n < 0 || k <= 0 || k % PTQ1_0_QK != 0) return ORC_ERR_SHAPE;
  int64_t nb = k / PTQ1_0_QK;
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (r * nb + b) * PTQ1_0_BYTES;
      float d = orc_float_from_half((uint16_t)(blk[26] | (blk[27] << 8)));
      for (int j = 0; j < PTQ1_0_QK; ++j) {
        int byte, tn;
        ptq1_0_place(j, &byte, &tn);
        w_out[r * k + b * PTQ1_0_QK + j] = (float)(ptq1_0_trit(blk[byte], tn) - 1) * d;
      }
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* scale4_gs32: symmetric 4-bit with an implicit zero point of 8              */
/* ------------------------------------------------------------------------ */

int orc_scale4_quantize(const float* w, int64_t n, int64_t k, uint8_t* blocks) {
  if (n < 0 || k <= 0 || k % SCALE4_QK != 0) return ORC_ERR_SHAPE;
  int64_t nb = k / SCALE4_QK;
  for (int64_t i = 0; i < n * k; ++i)
    if (!isfinite(w[i])) return ORC_ERR_NONFINITE;
  int status = ORC_OK;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* wb = w + r * k + b * SCALE4_QK;
      uint8_t* out = blocks + (r * nb + b) * SCALE4_BYTES;
      /* the weight of largest magnitude, with its sign (the first on a tie) */
      float m = 0.0f;
      for (int j = 0; j < SCALE4_QK; ++j)
        if (fabsf(wb[j]) > fabsf(m)) m = wb[j];
      float d = m / -8.0f; /* fp32 quotient, then fp16 */
      uint16_t dh = orc_half_from_float(d);
      if ((dh & 0x7C00) == 0x7C00) {
#pragma omp atomic write
        status = ORC_ERR_RANGE;
      }
      float df = orc_float_from_half(dh); /* quantize against the fp16-rounded scale */
      memset(out, 0, SCALE4_BYTES);
      out[0] = (uint8_t)(dh & 0xFF);
      out[1] = (uint8_t)(dh >> 8);
      for (int j = 0; j < SCALE4_QK; ++j) {
        long q = 8;
        if (df != 0.0f) {
          q = lround((double)wb[j] / (double)df) + 8;
          if (q > 15) q = 15;
          if (q < 0) q = 0;
        }
        out[2 + j / 2] |= (uint8_t)(q << (4 * (j % 2)));
      }
    }
  }
  return status;
}

int orc_scale4_dequant(const uint8_t* blocks, int64_t n, int64_t k, float* w_out) {
  if (n < 0 || k <= 0 || k % SCALE4_QK != 0) return ORC_ERR_SHAPE;
  int64_t nb = k / SCALE4_QK;
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (r * nb + b) * SCALE4_BYTES;
      float d = orc_float_from_half((uint16_t)(blk[0] | (blk[1] << 8)));
      for (int j = 0; j < SCALE4_QK; ++j) {
        int q = (blk[2 + j / 2] >> (4 * (j % 2))) & 15;
        w_out[r * k + b * SCALE4_QK + j] = (float)(q - 8) * d;
      }
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Hadamard rotation                                                          */
/* ------------------------------------------------------------------------ */

static int popcount64(uint64_t v) {
  int c = 0;
  while (v) {
    c += (int)(v & 1);
    v >>= 1;
  }
  return c;
}

static int is_pow2(int64_t n) { return n > 0 && (n & (n - 1)) == 0; }

int orc_hadamard(int32_t n, double* h_out) {
  if (!is_pow2(n)) return ORC_ERR_SHAPE;
  for (int32_t r = 0; r < n; ++r)
    for (int32_t c = 0; c < n; ++c) h_out[(int64_t)r * n + c] = (popcount64((uint64_t)(r & c)) & 1) ? -1.0 : 1.0;
  return ORC_OK;
}

int orc_rotate_rows(const float* in, int64_t rows, int64_t k, int32_t n, double* out64, float* out32) {
  return orc_rotate_rows_signed(in, rows, k, n, 0, out64, out32);
}

int orc_rotate_rows_signed(const float* in, int64_t rows, int64_t k, int32_t n, const int8_t* signs, double* out64,
                           float* out32) {
  if (!is_pow2(n) || rows < 0 || k <= 0 || k % n != 0) return ORC_ERR_SHAPE;
  if (signs)
    for (int64_t c = 0; c < k; ++c)
      if (signs[c] != 1 && signs[c] != -1) return ORC_ERR_SHAPE;
  const double inv_sqrt_n = 1.0 / sqrt((double)n);
  int64_t nblk = k / n;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nblk; ++b) {
      const float* v = in + r * k + b * n;
      const int8_t* sg = signs ? signs + b * n : 0;
      for (int32_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int32_t c = 0; c < n; ++c) {
          double h = (popcount64((uint64_t)(i & c)) & 1) ? -1.0 : 1.0;
          double xc = sg ? (double)sg[c] * (double)v[c] : (double)v[c];
          s += h * xc;
        }
        double o = inv_sqrt_n * s;
        int64_t at = r * k + b * n + i;
        if (out64) out64[at] = o;
        if (out32) out32[at] = (float)o;
      }
    }
  }
  return ORC_OK;
}

/* The inverse of the signed rotation, e = R^T z = S (H_n z) / sqrt(n) per
 * n-block: the transform first, then the sign flip (the Bonsai page, section
 * 4.2, embedding inverse), with the explicit FP64 matrix. */
int orc_rotate_rows_inverse(const float* in, int64_t rows, int64_t k, int32_t n, const int8_t* signs, double* out64) {
  if (!is_pow2(n) || rows < 0 || k <= 0 || k % n != 0) return ORC_ERR_SHAPE;
  if (signs)
    for (int64_t c = 0; c < k; ++c)
      if (signs[c] != 1 && signs[c] != -1) return ORC_ERR_SHAPE;
  const double inv_sqrt_n = 1.0 / sqrt((double)n);
  int64_t nblk = k / n;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nblk; ++b) {
      const float* v = in + r * k + b * n;
      for (int32_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int32_t c = 0; c < n; ++c) {
          double h = (popcount64((uint64_t)(i & c)) & 1) ? -1.0 : 1.0;
          s += h * (double)v[c];
        }
        double o = inv_sqrt_n * s;
        if (signs) o *= (double)signs[b * n + i];
        out64[r * k + b * n + i] = o;
      }
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* GEMV in FP64                                                               */
/* ------------------------------------------------------------------------ */

int orc_gemv_f64(const float* w, int64_t n, int64_t k, const double* x, const int64_t* rows, int64_t nrows,
                 int32_t rows_are_packed, double* y, double* absdot) {
  if (n < 0 || k <= 0) return ORC_ERR_SHAPE;
  if (rows == NULL) nrows = n;
  for (int64_t t = 0; t < nrows; ++t) {
    int64_t r = rows ? rows[t] : t;
    if (r < 0 || r >= n) return ORC_ERR_SHAPE;
  }
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < nrows; ++t) {
    int64_t r = rows ? rows[t] : t;
    const float* wr = w + (rows_are_packed ? t : r) * k;
    double s = 0.0, a = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      double p = (double)wr[j] * x[j];
      s += p;
      a += fabs(p);
    }
    y[t] = s;
    absdot[t] = a;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Array forms of the binary16 conversions, for the tests.                    */
/* ------------------------------------------------------------------------ */

void orc_half_from_float_array(const float* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_half_from_float(in[i]);
}

void orc_float_from_half_array(const uint16_t* in, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_float_from_half(in[i]);
}
