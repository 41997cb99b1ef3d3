/*
 * Seeded, counter-based generators for the synthetic MoE FFN workloads.
 *
 * This file holds no arithmetic of the MoE layer itself: it only draws the
 * layer's inputs (activations, router weight and bias, expert weights in bf16
 * or grouped Int4 form).  Both the CPU oracle side and the GPU side take their
 * inputs from here, so the two never disagree about what the inputs are.
 *
 * Every element is a pure function of (seed, tensor id, element index):
 *
 *   draw(seed, tid, n) = mix64(stream(seed, tid) + (n + 1) * GAMMA)
 *   stream(seed, tid)  = mix64(mix64(seed ^ SEED_SALT) ^ tid)
 *
 * where mix64 is the SplitMix64 output function (Steele, Lea, Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014) and GAMMA is
 * its golden-ratio increment.  Any sub-range of a tensor (one expert's slab,
 * one redrawn token row) can therefore be regenerated on its own.
 *
 * Normals use the Box-Muller transform on draw pairs (2m, 2m+1): element 2m
 * takes the cosine branch and element 2m+1 the sine branch.  Values are
 * formed in double precision, then rounded to the storage type with
 * round-to-nearest-even.
 *
 * Built with -ffp-contract=off so that no fused multiply-add changes the
 * double-precision values between compilers or CPU architectures.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL
#define SEED_SALT 0x5DEECE66DULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_of(uint64_t seed, uint64_t tid) {
  return mix64(mix64(seed ^ SEED_SALT) ^ tid);
}

static inline uint64_t draw(uint64_t base, uint64_t n) {
  return mix64(base + (n + 1ULL) * GAMMA);
}

/* uniform in [0, 1) with 53 random bits */
static inline double unit_co(uint64_t r) { return (double)(r >> 11) * 0x1.0p-53; }
/* uniform in (0, 1] with 53 random bits */
static inline double unit_oc(uint64_t r) { return ((double)(r >> 11) + 1.0) * 0x1.0p-53; }

static inline double normal_at(uint64_t base, uint64_t i) {
  const uint64_t m = i >> 1;
  const double u1 = unit_oc(draw(base, 2 * m));
  const double u2 = unit_co(draw(base, 2 * m + 1));
  const double r = sqrt(-2.0 * log(u1));
  const double th = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(th) : r * cos(th);
}

/* float -> bf16 bits, round to nearest even (NaN not produced here) */
static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* out[j] = bf16(std * N(0,1)) for elements start .. start+n-1 */
void syn_normal_bf16(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n,
                     double std_dev, uint16_t* out) {
  const uint64_t base = stream_of(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)n; ++j)
    out[j] = f32_to_bf16((float)(std_dev * normal_at(base, start + (uint64_t)j)));
}

/* out[j] = float(mean + std * N(0,1)) */
void syn_normal_f32(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n,
                    double mean, double std_dev, float* out) {
  const uint64_t base = stream_of(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)n; ++j)
    out[j] = (float)(mean + std_dev * normal_at(base, start + (uint64_t)j));
}

/* out[j] = bf16(U(lo, hi)) */
void syn_uniform_bf16(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n,
                      double lo, double hi, uint16_t* out) {
  const uint64_t base = stream_of(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)n; ++j) {
    const double u = unit_co(draw(base, start + (uint64_t)j));
    out[j] = f32_to_bf16((float)(lo + (hi - lo) * u));
  }
}

/* Packed 4-bit codes, uniform on 0..15.  Byte j holds code 2j (of the whole
 * tensor's element numbering, counted from `start_byte`*2) in its low nibble
 * and code 2j+1 in its high nibble.  Each code takes the top 4 bits of its own
 * draw, so the packing does not change which value an element gets. */
void syn_codes_u4(uint64_t seed, uint64_t tid, uint64_t start_byte, uint64_t n_bytes,
                  uint8_t* out) {
  const uint64_t base = stream_of(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)n_bytes; ++j) {
    const uint64_t e = 2 * (start_byte + (uint64_t)j);
    const uint8_t lo = (uint8_t)(draw(base, e) >> 60);
    const uint8_t hi = (uint8_t)(draw(base, e + 1) >> 60);
    out[j] = (uint8_t)(lo | (hi << 4));
  }
}

/* Raw 64-bit draws, exposed so tests can check the generator against the
 * published SplitMix64 reference sequence. */
void syn_raw(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n, uint64_t* out) {
  const uint64_t base = stream_of(seed, tid);
  for (uint64_t j = 0; j < n; ++j) out[j] = draw(base, start + j);
}

/* The SplitMix64 sequence itself: state starts at `state`, each output adds
 * GAMMA then mixes.  Used only to pin mix64/GAMMA to the published values. */
void syn_splitmix64_seq(uint64_t state, uint64_t n, uint64_t* out) {
  for (uint64_t j = 0; j < n; ++j) {
    state += GAMMA;
    out[j] = mix64(state);
  }
}
