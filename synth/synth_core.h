/* synth_core.h -- seeded, counter-based synthetic input generator.
 *
 * This module only makes input data. It holds none of the shard step's
 * arithmetic (no sums of gradients, no optimizer update, no rounding cast):
 * every value is produced from integers, exactly one IEEE double multiply and
 * a truncation of the resulting bit pattern toward zero. The same source is
 * compiled for the host (gcc) and for the device (nvcc), so both produce the
 * same bits for the same (seed, stream, index).
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used as a counter-based hash: draw j of
 * element i of a stream is mix64(key + (8*i + j + 1) * GAMMA), i.e. position
 * 8*i + j + 1 of the SplitMix64 sequence started at `key`.
 *
 * Distributions:
 *   normal   : Irwin-Hall sum of twelve 21-bit uniforms, centred and scaled to
 *              unit variance (the classic "sum of 12 uniforms minus 6"
 *              approximation of N(0,1), support +-6 sigma), times sigma;
 *   |normal| : absolute value of the above;
 *   uniform  : symmetric uniform on (-a, a) from a 53-bit draw.
 * An optional "outlier" selector (an independent stream) multiplies about one
 * element in `outlier_mod` by a second scale.
 *
 * Output formats: bf16, fp16 (bit patterns, uint16) and fp32 (uint32). The
 * double value is truncated toward zero onto the target format's grid,
 * including fp16/fp32 subnormals, so no rounding mode is involved.
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define SYNTH_FN static __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ull

enum { SYNTH_NORMAL = 0, SYNTH_ABS_NORMAL = 1, SYNTH_UNIFORM = 2 };
enum { SYNTH_FMT_BF16 = 0, SYNTH_FMT_FP16 = 1, SYNTH_FMT_FP32 = 2 };

typedef struct synth_spec {
  uint64_t seed;
  uint64_t stream;         /* packed (kind, rank, step) chosen by the caller */
  uint64_t outlier_stream; /* stream of the outlier selector */
  double scale;            /* normal: sigma * 2^-22 ; uniform: a * 2^-53 */
  double outlier_scale;    /* scale used where the selector fires */
  uint32_t outlier_mod;    /* 0: no outliers; else element i is an outlier when sel % mod == 0 */
  int32_t dist;            /* SYNTH_NORMAL / SYNTH_ABS_NORMAL / SYNTH_UNIFORM */
  int32_t fmt;             /* SYNTH_FMT_* */
  int32_t pad_;
} synth_spec;

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

SYNTH_FN uint64_t synth_key(uint64_t seed, uint64_t stream) {
  return synth_mix64(synth_mix64(seed ^ 0xD1B54A32D192ED03ull) + stream * SYNTH_GAMMA);
}

SYNTH_FN uint64_t synth_draw(uint64_t key, uint64_t i, uint32_t j) {
  return synth_mix64(key + (i * 8u + (uint64_t)j + 1u) * SYNTH_GAMMA);
}

/* Centred Irwin-Hall integer: 2*S - 12*(2^21-1), S = sum of twelve 21-bit
 * uniforms. Its standard deviation is 2^22 (to within 2^-42 relative). */
SYNTH_FN int64_t synth_irwin_hall(uint64_t key, uint64_t i) {
  const uint64_t m21 = (1ull << 21) - 1u;
  int64_t s = 0;
  for (uint32_t j = 0; j < 4; ++j) {
    uint64_t d = synth_draw(key, i, j);
    s += (int64_t)(d & m21) + (int64_t)((d >> 21) & m21) + (int64_t)((d >> 42) & m21);
  }
  return 2 * s - 12 * (int64_t)m21;
}

/* Symmetric odd integer in (-2^53, 2^53) from one 53-bit draw. */
SYNTH_FN int64_t synth_sym53(uint64_t key, uint64_t i) {
  int64_t d = (int64_t)(synth_draw(key, i, 0) >> 11);
  return 2 * d - (int64_t)((1ull << 53) - 1u);
}

/* Truncation toward zero of a double onto the fp32 grid (bit pattern). */
SYNTH_FN uint32_t synth_trunc_f32(double x) {
  uint64_t b;
  memcpy(&b, &x, sizeof b);
  uint32_t sign = (uint32_t)(b >> 63) << 31;
  int e = (int)((b >> 52) & 0x7FF);
  uint64_t man = b & ((1ull << 52) - 1u);
  if (e == 0) return sign;
  int ue = e - 1023;
  if (ue > 127) return sign | 0x7F7FFFFFu;
  if (ue >= -126) return sign | ((uint32_t)(ue + 127) << 23) | (uint32_t)(man >> 29);
  int sh = 52 - (ue + 149);
  if (sh >= 64) return sign;
  return sign | (uint32_t)((man | (1ull << 52)) >> sh);
}

/* Truncation toward zero onto the fp16 grid (bit pattern). */
SYNTH_FN uint16_t synth_trunc_f16(double x) {
  uint64_t b;
  memcpy(&b, &x, sizeof b);
  uint16_t sign = (uint16_t)((b >> 63) << 15);
  int e = (int)((b >> 52) & 0x7FF);
  uint64_t man = b & ((1ull << 52) - 1u);
  if (e == 0) return sign;
  int ue = e - 1023;
  if (ue > 15) return (uint16_t)(sign | 0x7BFFu);
  if (ue >= -14) return (uint16_t)(sign | ((uint32_t)(ue + 15) << 10) | (uint32_t)(man >> 42));
  int sh = 52 - (ue + 24);
  if (sh >= 64) return sign;
  return (uint16_t)(sign | (uint16_t)((man | (1ull << 52)) >> sh));
}

/* The double value of element i before it is put on the target grid. */
SYNTH_FN double synth_value(const synth_spec* s, uint64_t key, uint64_t sel_key, uint64_t i) {
  double scale = s->scale;
  if (s->outlier_mod != 0u && synth_draw(sel_key, i, 0) % s->outlier_mod == 0u) scale = s->outlier_scale;
  if (s->dist == SYNTH_UNIFORM) return (double)synth_sym53(key, i) * scale;
  int64_t z = synth_irwin_hall(key, i);
  if (s->dist == SYNTH_ABS_NORMAL && z < 0) z = -z;
  return (double)z * scale;
}

/* Bit pattern of element i in the spec's format (low 16 bits for bf16/fp16). */
SYNTH_FN uint32_t synth_bits(const synth_spec* s, uint64_t key, uint64_t sel_key, uint64_t i) {
  double x = synth_value(s, key, sel_key, i);
  if (s->fmt == SYNTH_FMT_FP32) return synth_trunc_f32(x);
  if (s->fmt == SYNTH_FMT_BF16) return synth_trunc_f32(x) >> 16;
  return synth_trunc_f16(x);
}

#endif /* SYNTH_CORE_H */
