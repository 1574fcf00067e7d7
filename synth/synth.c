/*
 * Seeded synthetic inputs for the BASTION draft-tree hot path.
 *
 * This module is shared by the checker (oracle) side and the CUDA side: it
 * produces input bytes only and holds none of the method's arithmetic (no
 * softmax, no ranking, no tree search, no argmax).
 *
 * Random numbers come from a counter-based construction on the splitmix64
 * mixing function (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; the finaliser constants are Vigna's published
 * splitmix64).  A draw is addressed by (seed, stream, index), so any element of
 * any tensor can be produced independently of thread count or order.
 *
 *   key(seed, stream) = mix(seed ^ mix(stream))
 *   u64(seed, stream, i) = mix(key + (i + 1) * GOLDEN)
 *   uniform = ((u64 >> 11) + 0.5) * 2^-53           in (0, 1), never 0 or 1
 *   normal  = Box-Muller on the uniform pair (2p, 2p+1), p = i >> 1:
 *             r = sqrt(-2 ln u1), theta = 2 pi u2,
 *             even i -> r cos(theta), odd i -> r sin(theta)
 *
 * bf16 values are produced from the double by one round-to-nearest-even step
 * (no intermediate float rounding).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* The published stepping form (state += GOLDEN, then mix), kept so a test can
 * check the mixing function against the generator's published output values. */
uint64_t synth_splitmix64_next(uint64_t *state) {
  *state += GOLDEN;
  return mix64(*state);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed ^ mix64(stream));
}

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t index) {
  return mix64(stream_key(seed, stream) + (index + 1) * GOLDEN);
}

static inline double u01_from(uint64_t x) {
  return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

double synth_uniform(uint64_t seed, uint64_t stream, uint64_t index) {
  return u01_from(synth_u64(seed, stream, index));
}

static inline double normal_at(uint64_t key, uint64_t i) {
  uint64_t p = i >> 1;
  double u1 = u01_from(mix64(key + (2 * p + 1) * GOLDEN));
  double u2 = u01_from(mix64(key + (2 * p + 2) * GOLDEN));
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(th) : r * cos(th);
}

double synth_normal(uint64_t seed, uint64_t stream, uint64_t index) {
  return normal_at(stream_key(seed, stream), index);
}

/* Round a double to the nearest bfloat16 (ties to even), returning its bits. */
uint16_t synth_f64_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isinf(a)) return sign | 0x7F80;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);                      /* a in [2^(e-1), 2^e) */
  int qexp = e - 8;                  /* 8 significant bits */
  if (qexp < -133) qexp = -133;      /* subnormal quantum 2^-133 */
  double n = nearbyint(ldexp(a, -qexp));  /* exact scaling, RNE */
  double y = ldexp(n, qexp);
  if (y > 3.3895313892515355e38) return sign | 0x7F80;  /* above max bf16 */
  float f = (float)y;                /* exact: y has <= 8 significant bits */
  uint32_t bits;
  memcpy(&bits, &f, 4);
  return sign | (uint16_t)((bits >> 16) & 0x7FFF);
}

/* out[i] = scale * normal(seed, stream, offset + i) for i in [0, n), as bf16. */
void synth_fill_normal_bf16(uint16_t *out, int64_t n, double scale, uint64_t seed,
                            uint64_t stream, int64_t offset) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static, 65536)
  for (int64_t i = 0; i < n; ++i)
    out[i] = synth_f64_to_bf16(scale * normal_at(key, (uint64_t)(offset + i)));
}

/* Same as above, rounded to float (one RNE step from the double). */
void synth_fill_normal_f32(float *out, int64_t n, double scale, uint64_t seed,
                           uint64_t stream, int64_t offset) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static, 65536)
  for (int64_t i = 0; i < n; ++i)
    out[i] = (float)(scale * normal_at(key, (uint64_t)(offset + i)));
}

/* Row-strided variant: rows x cols elements, row r starting at out + r*ld,
 * element (r, c) drawn at index offset + r*cols + c. */
void synth_fill_normal_rows_bf16(uint16_t *out, int64_t rows, int64_t cols, int64_t ld,
                                 double scale, uint64_t seed, uint64_t stream,
                                 int64_t offset) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static, 4)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * ld + c] =
          synth_f64_to_bf16(scale * normal_at(key, (uint64_t)(offset + r * cols + c)));
}

void synth_fill_normal_rows_f32(float *out, int64_t rows, int64_t cols, int64_t ld,
                                double scale, uint64_t seed, uint64_t stream,
                                int64_t offset) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static, 4)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * ld + c] = (float)(scale * normal_at(key, (uint64_t)(offset + r * cols + c)));
}

/* Fill n uniforms in (0,1) (double), for small per-request draws. */
void synth_fill_uniform(double *out, int64_t n, uint64_t seed, uint64_t stream,
                        int64_t offset) {
  uint64_t key = stream_key(seed, stream);
  for (int64_t i = 0; i < n; ++i)
    out[i] = u01_from(mix64(key + ((uint64_t)(offset + i) + 1) * GOLDEN));
}
