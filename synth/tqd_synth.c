/*
 * Seeded synthetic inputs for the Q8_0 greedy-decode path.
 *
 * This module builds inputs only: a counter-based PRNG (splitmix64), an
 * approximately normal draw, f32 -> f16 / bf16 encoding, the Q8_0 quantizer
 * that turns a float weight block into the 34-byte block the decoder reads,
 * uniform token ids and uniform fills.  It contains none of the decode step's
 * arithmetic (no dequantisation, no matvec, norm, rotation, attention or
 * argmax): both the oracle and the CUDA library consume the bytes it writes.
 *
 * Definitions (all bit-reproducible on any IEEE-754 host):
 *   mix64(z)          splitmix64 finaliser (Steele, Lea, Flood, "Fast
 *                     splittable pseudorandom number generators", 2014).
 *   stream(seed, t)   = mix64(seed ^ (0xD1B54A32D192ED03 * (t + 1)))
 *   draw(s, k)        = mix64(s + (k + 1) * 0x9E3779B97F4A7C15)
 *   normal element i  : words draw(s,3i), draw(s,3i+1), draw(s,3i+2) give
 *                       twelve 16-bit uniforms u; S = sum(u);
 *                       z = (2 S - 12*65535) / 131072   (exact in f64;
 *                       mean 0, variance 1 - 2^-32: Irwin-Hall(12), tails
 *                       cut at +-6), value = (float)(mean + sigma * z).
 *   Q8_0 block        : 32 consecutive row elements w; amax = max|w| (f32);
 *                       d = amax / 127 (f32); scale = f16(d) rounded to
 *                       nearest-even; q = clamp(rint(w / d), -127, 127)
 *                       with w / d in f32 (q = 0 when d == 0); bytes =
 *                       scale little-endian, then the 32 quants.
 *   token id          : draw(stream(seed, 0x10000 + seq), i) % vocab.
 *   uniform element i : lo + (hi - lo) * (draw(s,i) >> 11) * 2^-53, to f32.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define TQS_GOLDEN 0x9E3779B97F4A7C15ULL
#define TQS_STREAM_MUL 0xD1B54A32D192ED03ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t tqs_stream(uint64_t seed, uint64_t tensor) {
  return mix64(seed ^ (TQS_STREAM_MUL * (tensor + 1)));
}

uint64_t tqs_draw(uint64_t stream, uint64_t k) {
  return mix64(stream + (k + 1) * TQS_GOLDEN);
}

/* Irwin-Hall(12) standard draw for element i of a stream, exact in f64. */
static inline double std_draw(uint64_t s, uint64_t i) {
  uint64_t sum = 0;
  for (int w = 0; w < 3; ++w) {
    uint64_t r = tqs_draw(s, 3 * i + (uint64_t)w);
    sum += (r & 0xFFFF) + ((r >> 16) & 0xFFFF) + ((r >> 32) & 0xFFFF) + (r >> 48);
  }
  return ((double)(2 * (int64_t)sum) - 12.0 * 65535.0) / 131072.0;
}

double tqs_std_normal(uint64_t stream, uint64_t i) { return std_draw(stream, i); }

uint16_t tqs_f32_to_f16(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) return (uint16_t)(sign | (ax > 0x7F800000u ? 0x7E00u : 0x7C00u));
  if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* >= 65520 rounds to inf */
  if (ax < 0x38800000u) {                                   /* below 2^-14: subnormal */
    if (ax <= 0x33000000u) return (uint16_t)sign;           /* <= 2^-25 rounds to 0 */
    uint32_t e = ax >> 23;
    uint32_t m = (ax & 0x7FFFFFu) | 0x800000u;
    uint32_t shift = 126u - e; /* value in units of 2^-24 is m >> shift */
    uint32_t q = m >> shift, rem = m & ((1u << shift) - 1u), half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (q & 1u))) q++;
    return (uint16_t)(sign | q);
  }
  uint32_t q = ((((ax >> 23) - 112u)) << 10) | ((ax & 0x7FFFFFu) >> 13);
  uint32_t rem = ax & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q++;
  return (uint16_t)(sign | q);
}

uint16_t tqs_f32_to_bf16(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  if ((x & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((x >> 16) | 0x40u);
  x += 0x7FFFu + ((x >> 16) & 1u);
  return (uint16_t)(x >> 16);
}

/* out[i] = (float)(mean + sigma * z_i) for the tensor's stream. */
void tqs_normal_f32(uint64_t seed, uint64_t tensor, int64_t n, double mean, double sigma,
                    float* out) {
  uint64_t s = tqs_stream(seed, tensor);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(mean + sigma * std_draw(s, (uint64_t)i));
}

/* Quantise 32 floats into one 34-byte Q8_0 block. */
void tqs_quantize_block(const float* w, uint8_t* blk) {
  float amax = 0.0f;
  for (int j = 0; j < 32; ++j) {
    float a = fabsf(w[j]);
    if (a > amax) amax = a;
  }
  float d = amax / 127.0f;
  uint16_t h = tqs_f32_to_f16(d);
  blk[0] = (uint8_t)(h & 0xFF);
  blk[1] = (uint8_t)(h >> 8);
  for (int j = 0; j < 32; ++j) {
    int q = 0;
    if (d != 0.0f) {
      float r = rintf(w[j] / d);
      q = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);
    }
    blk[2 + j] = (uint8_t)(int8_t)q;
  }
}

/* A [rows x cols] matrix of N(0, sigma) weights (row-major element order)
 * quantised to Q8_0: rows * cols/32 blocks of 34 bytes, row after row. */
int tqs_q8_0_matrix(uint64_t seed, uint64_t tensor, int64_t rows, int64_t cols, double sigma,
                    uint8_t* out) {
  if (cols % 32 != 0 || rows < 0) return -1;
  uint64_t s = tqs_stream(seed, tensor);
  int64_t bpr = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    float w[32];
    for (int64_t b = 0; b < bpr; ++b) {
      for (int j = 0; j < 32; ++j)
        w[j] = (float)(sigma * std_draw(s, (uint64_t)(r * cols + b * 32 + j)));
      tqs_quantize_block(w, out + (r * bpr + b) * 34);
    }
  }
  return 0;
}

/* The same N(0, sigma) matrix rounded to bf16 (nearest-even). */
int tqs_bf16_matrix(uint64_t seed, uint64_t tensor, int64_t rows, int64_t cols, double sigma,
                    uint16_t* out) {
  if (rows < 0 || cols < 0) return -1;
  uint64_t s = tqs_stream(seed, tensor);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] =
          tqs_f32_to_bf16((float)(sigma * std_draw(s, (uint64_t)(r * cols + c))));
  return 0;
}

void tqs_token_ids(uint64_t seed, int64_t seq, int64_t n, int64_t vocab, int32_t* out) {
  uint64_t s = tqs_stream(seed, 0x10000u + (uint64_t)seq);
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(tqs_draw(s, (uint64_t)i) % (uint64_t)vocab);
}

void tqs_uniform_f32(uint64_t seed, uint64_t tensor, int64_t n, double lo, double hi, float* out) {
  uint64_t s = tqs_stream(seed, tensor);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double u = (double)(tqs_draw(s, (uint64_t)i) >> 11) * (1.0 / 9007199254740992.0);
    out[i] = (float)(lo + (hi - lo) * u);
  }
}
