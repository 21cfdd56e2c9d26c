/*
 * Seeded, counter-based synthetic input generator (weights, KV cache, hidden
 * states, token ids).  This header holds the generator only: none of the
 * tensor-parallel method's arithmetic lives here.  Both the host fill
 * (synth_host.c) and the device fill (synth_cuda.cu) include it, so a value is
 * a pure function of (seed, tensor id, flat index) on either side.
 *
 * Definition
 *   key(seed, tid)   = SM(SM(seed) ^ tid)             SM = SplitMix64 finaliser
 *                                                      applied to state+gamma
 *   bits(i)          = mix(key + (i + 1) * gamma)     the i-th SplitMix64 output
 *   normal-ish(i)    = Irwin-Hall(4) of the four 16-bit fields of bits(i),
 *                      centred and scaled to unit variance, times sigma,
 *                      rounded once to bf16 (round to nearest, ties to even)
 *   uniform int(i)   = ((bits(i) >> 32) * n) >> 32    in [0, n)
 *
 * SplitMix64 is the generator of Steele, Lea and Flood (OOPSLA 2014) with the
 * constants Vigna published for it.  The Irwin-Hall(4) law is bounded at
 * +-2*sqrt(3) sigma; it stands in for N(0, sigma^2).
 */
#ifndef SYNTH_DEF_H
#define SYNTH_DEF_H

#include <stdint.h>
#include <math.h>

#ifdef __CUDACC__
#define SYNTH_HD __host__ __device__ __forceinline__
#else
#define SYNTH_HD static inline
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

SYNTH_HD uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

SYNTH_HD uint64_t synth_key(uint64_t seed, uint64_t tensor_id) {
  return synth_mix64(synth_mix64(seed + SYNTH_GAMMA) ^ tensor_id);
}

SYNTH_HD uint64_t synth_bits(uint64_t key, uint64_t i) {
  return synth_mix64(key + (i + 1ULL) * SYNTH_GAMMA);
}

/* Unit-variance Irwin-Hall(4) sample times `scale` (scale = sigma, passed in
 * by the caller so both sides multiply by the identical double). */
SYNTH_HD double synth_normalish(uint64_t b, double scale_sqrt3) {
  int64_t s = (int64_t)(b & 0xFFFF) + (int64_t)((b >> 16) & 0xFFFF) +
              (int64_t)((b >> 32) & 0xFFFF) + (int64_t)((b >> 48) & 0xFFFF);
  double centred = (double)(s - 131070); /* exact: |s - 131070| < 2^18 */
  double x = centred * 0x1p-16;          /* exact: power-of-two scaling */
  return x * scale_sqrt3;                /* one rounding */
}

/* double -> bf16 bits, round to nearest, ties to even, in one step (no
 * intermediate float rounding).  Finite inputs only. */
SYNTH_HD uint16_t synth_double_to_bf16(double x) {
  if (x == 0.0) return signbit(x) ? (uint16_t)0x8000 : (uint16_t)0;
  int e;
  (void)frexp(x, &e);          /* |x| in [2^(e-1), 2^e) */
  int q = e - 1 - 7;           /* quantum of an 8-significant-bit value */
  if (q < -133) q = -133;      /* bf16 subnormal quantum */
  double r = rint(ldexp(x, -q)); /* exact scaling, then RNE to an integer */
  double y = ldexp(r, q);        /* exactly representable in bf16 (or 2^128) */
  float f = (float)y;            /* exact, or +-inf on overflow */
  union { float f; uint32_t u; } cv;
  cv.f = f;
  return (uint16_t)(cv.u >> 16);
}

SYNTH_HD uint16_t synth_normal_bf16(uint64_t key, uint64_t i, double scale_sqrt3) {
  return synth_double_to_bf16(synth_normalish(synth_bits(key, i), scale_sqrt3));
}

SYNTH_HD int32_t synth_uniform_int(uint64_t key, uint64_t i, uint32_t n) {
  return (int32_t)(((synth_bits(key, i) >> 32) * (uint64_t)n) >> 32);
}

#endif
