/*
 * FP64 CPU oracle of the quantized weight-streaming GEMV.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this code; the product library never
 * links, calls or falls back to it, and it shares no code with the product.
 *
 * It is a plain, slow restatement of the definitions on the pages:
 *
 *  - Q8_0 ("Kipp Architecture", section "Weight quantization"): blocks of 32
 *    weights along K, an fp16 scale d and int8 codes q, value d*q; the
 *    converter quantizes against the fp16-rounded scale.  Block = 2 B of d
 *    (little endian) followed by 32 int8 codes (34 B; 136 B per 128-dim row
 *    in "Kipp Benchmarks", Quantized KV cache bullet).
 *  - PQ2_0 ("Bonsai 2 27B - ternary g128 + blockwise Hadamard", section 3.1):
 *    128-weight blocks of 34 B, fp16 d first, then 32 bytes of 2-bit codes;
 *    element j sits in byte j/4 at bit offset 2*(j%4); code q in {0,1,2}
 *    has value (q-1)*d; the quantiser takes d = max|w| over the group and
 *    q = round(w/d) + 1.
 *  - The rotation (same page, sections 4.1 and 4.2): R = (1/sqrt(n)) * H_n,
 *    H_n the natural-order Sylvester matrix H[r][c] = (-1)^popcount(r & c),
 *    applied block-diagonally along K; the stored weight is W' = W R^T
 *    (rotate, then quantize) and the activation gets x' = R x before the
 *    product.  n = 128 with S = I by default; orc_rotate_rows_signed takes
 *    the page's general form, any power-of-two n (1024 on the page) and a
 *    +-1 sign per position of K applied before the transform.
 *
 * Readings where the pages are silent:
 *  - round() is round-half-away-from-zero (C round), decided on the FP64
 *    ratio of two floats, which is exact enough to see every tie;
 *  - the Q8_0 scale is the fp32 quotient amax/127, then rounded to fp16 with
 *    round-to-nearest-even; codes are clamped to [-127, 127];
 *  - a block whose fp16 scale is zero gets codes 0 (Q8_0) or 1 (PQ2_0);
 *  - R w is evaluated as (1/sqrt(n)) * (H w): the sum in FP64, one FP64
 *    multiply, then (for stored weights) one rounding to fp32.
 *
 * Every output of the GEMV is the FP64 value of the finite sum
 * sum_j deq(W)_ij * x_j (x' for PQ2_0), summed in index order, together with
 * sum_j |deq(W)_ij * x_j|, the scale of the acceptance bound.
 */
#ifndef KQ_ORACLE_H
#define KQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_ERR_SHAPE = 1, ORC_ERR_NONFINITE = 2, ORC_ERR_RANGE = 3 };

/* IEEE 754 binary16 <-> binary32, round to nearest even (overflow -> inf). */
uint16_t orc_half_from_float(float f);
float orc_float_from_half(uint16_t h);
void orc_half_from_float_array(const float* in, int64_t n, uint16_t* out);
void orc_float_from_half_array(const uint16_t* in, int64_t n, float* out);

/* Q8_0: w is n x k row-major fp32, k % 32 == 0; blocks gets n*k/32 blocks of 34 B. */
int orc_q8_0_quantize(const float* w, int64_t n, int64_t k, uint8_t* blocks);
int orc_q8_0_dequant(const uint8_t* blocks, int64_t n, int64_t k, float* w_out);

/* PQ2_0: w_rot is the already rotated n x k matrix, k % 128 == 0; n*k/128 blocks of 34 B. */
int orc_pq2_0_quantize(const float* w_rot, int64_t n, int64_t k, uint8_t* blocks);
int orc_pq2_0_dequant(const uint8_t* blocks, int64_t n, int64_t k, float* w_out);

/* PTQ1_0 ("Bonsai 2 27B", section 3.2): the trits and the fp16 scale of
 * PQ2_0 (value (t-1)*d, d = max|w|, t = round(w/d) + 1) packed in base 3 into
 * 28-byte blocks of 128: qs[24] with five trits per byte, qh[2] with four,
 * then d (last, unlike PQ2_0).  A byte holds q = ceil(256 v / 243), v the
 * trits as a base-3 number with the first trit most significant (a qh byte's
 * absent fifth trit taken as 0); trit n is ((q 3^n) mod 256) * 3 / 256,
 * rounded down.  Element order, from the page's table: 0-79 are trit e/16 of
 * qs[e%16], 80-119 trit (e-80)/8 of qs[16+(e-80)%8], 120-127 trit (e-120)/2
 * of qh[(e-120)%2].  w_rot is the already rotated n x k matrix, k % 128 == 0. */
int orc_ptq1_0_quantize(const float* w_rot, int64_t n, int64_t k, uint8_t* blocks);
int orc_ptq1_0_dequant(const uint8_t* blocks, int64_t n, int64_t k, float* w_out);
/* The byte rule and the trit rule on their own (trits: five values 0..2). */
int orc_ptq1_0_encode_byte(const int32_t* trits);
int orc_ptq1_0_decode_trit(int32_t q, int32_t n);

/* scale4_gs32 ("Kipp Benchmarks", section "Scale-only 4-bit (scale4_gs32)"):
 * 32-weight groups of 16 packed nibbles plus one fp16 scale (18 bytes,
 * 4.5 bits per weight), w = d (q - 8), q in 0..15; the converter takes the
 * weight of largest magnitude m with its sign and d = m / -8 (Q4_0-class),
 * and quantizes against the fp16-rounded scale.  Readings where the page is
 * silent: the fp32 quotient m / -8 rounded to fp16 to nearest even; the first
 * weight on a tie of magnitudes; q = round-half-away-from-zero(w / d) + 8
 * clamped to [0, 15]; a group whose fp16 scale is zero gets q = 8; the scale
 * first (bytes 0-1, little endian), then element j in byte 2 + j/2 at bit
 * offset 4 (j % 2), the same nibble order rule as the PQ2_0 crumbs. */
int orc_scale4_quantize(const float* w, int64_t n, int64_t k, uint8_t* blocks);
int orc_scale4_dequant(const uint8_t* blocks, int64_t n, int64_t k, float* w_out);

/* Unnormalised Sylvester Hadamard matrix, n x n row-major, entries +-1. */
int orc_hadamard(int32_t n, double* h_out);

/* Blockwise rotation of each row: out = (1/sqrt(n)) * (H_n block) per n-block
 * of K.  out64 (may be NULL) gets the FP64 values, out32 (may be NULL) the
 * same values rounded once to fp32. */
int orc_rotate_rows(const float* in, int64_t rows, int64_t k, int32_t n, double* out64, float* out32);

/* The same with a diagonal sign matrix first (the Bonsai page, section 4.1:
 * R = (1/sqrt(n)) H_n S, S = diag(signs), one +-1 per position of K; sign
 * flip, then the transform, section 4.2).  signs == NULL is S = I; an entry
 * other than +1 or -1 is ORC_ERR_SHAPE. */
int orc_rotate_rows_signed(const float* in, int64_t rows, int64_t k, int32_t n, const int8_t* signs, double* out64,
                           float* out32);

/* The inverse rotation e = R^T z = S (H_n z) / sqrt(n) per n-block (the
 * Bonsai page, section 4.2: the embedding table stores R e per row; after
 * the gather, transform first, then the sign flip).  FP64 out. */
int orc_rotate_rows_inverse(const float* in, int64_t rows, int64_t k, int32_t n, const int8_t* signs, double* out64);

/* y_i = sum_j w_ij x_j and absdot_i = sum_j |w_ij x_j| in FP64 for the listed
 * rows (rows == NULL: all n rows, in order); w holds the n x k matrix (or
 * just the listed rows when rows_are_packed != 0). */
int orc_gemv_f64(const float* w, int64_t n, int64_t k, const double* x, const int64_t* rows, int64_t nrows,
                 int32_t rows_are_packed, double* y, double* absdot);

/* Threads the row loops may use (OpenMP), for reporting. */
int orc_max_threads(void);
void orc_set_threads(int n);

#ifdef __cplusplus
}
#endif

#endif /* KQ_ORACLE_H */
