/* Host fill for the synthetic input generator defined in synth_def.h.
 * Multi-threaded with OpenMP; every element is an independent function of its
 * flat index, so the result does not depend on the thread count. */
#include <stddef.h>
#include "synth_def.h"

/* out[j] = bf16 sample for flat index start + j, j in [0, count). */
void synth_fill_normal_bf16(uint16_t* out, uint64_t seed, uint64_t tensor_id,
                            uint64_t start, uint64_t count, double scale_sqrt3) {
  const uint64_t key = synth_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)count; ++j)
    out[j] = synth_normal_bf16(key, start + (uint64_t)j, scale_sqrt3);
}

/* out[j] = uniform integer in [0, n) for flat index start + j. */
void synth_fill_uniform_i32(int32_t* out, uint64_t seed, uint64_t tensor_id,
                            uint64_t start, uint64_t count, uint32_t n) {
  const uint64_t key = synth_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)count; ++j)
    out[j] = synth_uniform_int(key, start + (uint64_t)j, n);
}
