/* synth_host.c -- host side of the seeded input generator (see synth_core.h).
 * Fills host arrays for a contiguous index range or for a list of indices. */
#include "synth_core.h"

static void store(const synth_spec* s, void* out, uint64_t k, uint32_t bits) {
  if (s->fmt == SYNTH_FMT_FP32) ((uint32_t*)out)[k] = bits;
  else ((uint16_t*)out)[k] = (uint16_t)bits;
}

int synth_fill_range(const synth_spec* s, uint64_t start, uint64_t count, void* out) {
  if (!s || (!out && count)) return 1;
  uint64_t key = synth_key(s->seed, s->stream);
  uint64_t sel = synth_key(s->seed, s->outlier_stream);
  #pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < (int64_t)count; ++k)
    store(s, out, (uint64_t)k, synth_bits(s, key, sel, start + (uint64_t)k));
  return 0;
}

int synth_fill_gather(const synth_spec* s, const uint64_t* idx, uint64_t count, void* out) {
  if (!s || ((!out || !idx) && count)) return 1;
  uint64_t key = synth_key(s->seed, s->stream);
  uint64_t sel = synth_key(s->seed, s->outlier_stream);
  #pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < (int64_t)count; ++k)
    store(s, out, (uint64_t)k, synth_bits(s, key, sel, idx[k]));
  return 0;
}

/* Raw integer draws, exposed so tests can check the generator's statistics. */
int64_t synth_irwin_hall_at(uint64_t seed, uint64_t stream, uint64_t i) {
  return synth_irwin_hall(synth_key(seed, stream), i);
}
