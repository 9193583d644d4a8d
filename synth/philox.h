/*
 * Seeded synthetic input generator, shared by the host generator (gen_host.c)
 * and its device twin (gen_device.cu).  It holds no arithmetic of the
 * quantized GEMV method: it only turns (seed, stream, element index) into a
 * float that is identical, bit for bit, on the CPU and on the GPU.
 *
 * Generator: Philox4x64-10, the counter-based generator of Salmon, Moraes,
 * Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11):
 * a 4x64-bit counter and a 2x64-bit key, ten rounds of two 64x64->128 bit
 * multiplies with the key bumped by the Weyl constants between rounds.
 *
 * Value: the Irwin-Hall sum of twelve uniform integers (the classic
 * "sum of 12 uniforms minus 6" normal approximation), each uniform drawn from
 * one 16-bit slice of the Philox output and mapped onto [0, range) by a
 * multiply-shift.  The centred integer sum m is returned as m * 2^-exp2, which
 * is exact in fp32 (|m| < 2^20), so every consumer sees the same bits and
 * every block sum of up to 128 such weights is exact in fp32 and fp64.
 *
 *   weights     range = 20972, exp2 = 20  ->  std 0.0200005 (about N(0, 0.02))
 *   activations range = 65536, exp2 = 16  ->  std 1.0       (about N(0, 1))
 *
 * Sample i of a stream uses counter (i, 0, 0, 0) and key (seed, stream).
 */
#ifndef SYNTH_PHILOX_H
#define SYNTH_PHILOX_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_HD __host__ __device__ __forceinline__
#else
#define SYNTH_HD static inline
#endif

#define SYNTH_PHILOX_M0 0xD2E7470EE14C6C93ULL
#define SYNTH_PHILOX_M1 0xCA5A826395121157ULL
#define SYNTH_PHILOX_W0 0x9E3779B97F4A7C15ULL
#define SYNTH_PHILOX_W1 0xBB67AE8584CAA73BULL

/* Distribution presets (see the header comment). */
#define SYNTH_W_RANGE 20972u
#define SYNTH_W_EXP2 20
#define SYNTH_X_RANGE 65536u
#define SYNTH_X_EXP2 16

SYNTH_HD void synth_mulhilo64(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo) {
#if defined(__CUDA_ARCH__)
  *lo = a * b;
  *hi = __umul64hi(a, b);
#else
  unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
  *lo = (uint64_t)p;
  *hi = (uint64_t)(p >> 64);
#endif
}

/* One Philox4x64-10 block: out = bijection_key(ctr). */
SYNTH_HD void synth_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
  uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t hi0, lo0, hi1, lo1;
    synth_mulhilo64(SYNTH_PHILOX_M0, x0, &hi0, &lo0);
    synth_mulhilo64(SYNTH_PHILOX_M1, x2, &hi1, &lo1);
    uint64_t y0 = hi1 ^ x1 ^ k0;
    uint64_t y2 = hi0 ^ x3 ^ k1;
    x0 = y0;
    x1 = lo1;
    x2 = y2;
    x3 = lo0;
    k0 += SYNTH_PHILOX_W0;
    k1 += SYNTH_PHILOX_W1;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

/* Centre of the twelve-uniform sum for a given range: 12 * (range - 1) / 2. */
SYNTH_HD int32_t synth_center(uint32_t range) { return (int32_t)(6u * (range - 1u)); }

/* Sample `index` of stream (seed, stream) as a float: m * 2^-exp2. */
SYNTH_HD float synth_sample(uint64_t seed, uint64_t stream, uint64_t index, uint32_t range, int exp2) {
  uint64_t ctr[4] = {index, 0, 0, 0};
  uint64_t key[2] = {seed, stream};
  uint64_t r[4];
  synth_philox4x64_10(ctr, key, r);
  uint32_t sum = 0;
  for (int w = 0; w < 3; ++w) {
    for (int s = 0; s < 4; ++s) {
      uint32_t slice = (uint32_t)((r[w] >> (16 * s)) & 0xFFFFu);
      sum += (uint32_t)(((uint64_t)slice * (uint64_t)range) >> 16);
    }
  }
  int32_t m = (int32_t)sum - synth_center(range);
  /* m fits in 21 bits, so the conversion and the power-of-two scaling are exact. */
  float scale = 1.0f;
  for (int e = 0; e < exp2; ++e) scale *= 0.5f;
  return (float)m * scale;
}

#endif /* SYNTH_PHILOX_H */
