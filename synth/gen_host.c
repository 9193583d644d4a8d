/*
 * Host side of the seeded synthetic input generator (see philox.h).
 * Built as synth/_build/libsynth_host.so and called through ctypes.
 */
#include <stdint.h>
#include "philox.h"

/* out[i] = sample(first_index + i) for i in [0, n). */
void synth_fill_host(float* out, int64_t n, uint64_t seed, uint64_t stream, uint64_t first_index,
                     uint32_t range, int32_t exp2) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    out[i] = synth_sample(seed, stream, first_index + (uint64_t)i, range, exp2);
  }
}

/* Raw generator block, exposed so that tests can check it against other
 * implementations of Philox4x64-10. */
void synth_philox_block(const uint64_t* ctr, const uint64_t* key, uint64_t* out) {
  synth_philox4x64_10(ctr, key, out);
}
