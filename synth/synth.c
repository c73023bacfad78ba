/*
 * Seeded synthetic inputs for the Qwen2-style prefill (weights, norm gains,
 * biases, prompt token ids).  This file holds no arithmetic of the forward
 * pass: it only turns (seed, stream, index) into numbers.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used as a counter-based hash, followed by
 * the Box-Muller transform (Box & Muller, Ann. Math. Stat. 1958) in double.
 *
 *   key(seed, stream) = mix(seed ^ mix(stream + 1))
 *   u64(seed, stream, i) = mix(key + i)
 *   normal(i): r1 = u64(2i), r2 = u64(2i+1),
 *              u1 = ((r1 >> 11) + 1) * 2^-53   in (0, 1]
 *              u2 = (r2 >> 11) * 2^-53          in [0, 1)
 *              z  = sqrt(-2 ln u1) * cos(2 pi u2)
 *              value = (float)(mean + std * z)
 *   id(i) = ((u64(i) >> 32) * vocab) >> 32     (multiply-shift range map)
 *
 * mix() is the SplitMix64 output function applied to (x + golden gamma).
 * Every value depends only on its own counter, so any sub-range can be
 * generated independently and in parallel with identical results.
 */
#include <stdint.h>
#include <math.h>

static uint64_t mix(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix(seed ^ mix(stream + 1));
}

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t i) {
  return mix(stream_key(seed, stream) + i);
}

/* out[j] = normal value of counter (first + j), j in [0, n). */
void synth_normal_f32(uint64_t seed, uint64_t stream, double mean, double std,
                      int64_t first, int64_t n, float* out) {
  const uint64_t key = stream_key(seed, stream);
  const double two_pi = 6.283185307179586476925286766559;
  const double inv53 = 1.0 / 9007199254740992.0; /* 2^-53 */
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) {
    const uint64_t i = (uint64_t)(first + j);
    const uint64_t r1 = mix(key + 2 * i);
    const uint64_t r2 = mix(key + 2 * i + 1);
    const double u1 = (double)((r1 >> 11) + 1) * inv53;
    const double u2 = (double)(r2 >> 11) * inv53;
    const double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
    out[j] = (float)(mean + std * z);
  }
}

/* out[j] = token id in [0, vocab) of counter (first + j). */
void synth_ids(uint64_t seed, uint64_t stream, int32_t vocab, int64_t first,
               int64_t n, int32_t* out) {
  const uint64_t key = stream_key(seed, stream);
  for (int64_t j = 0; j < n; ++j) {
    const uint64_t r = mix(key + (uint64_t)(first + j));
    out[j] = (int32_t)(((r >> 32) * (uint64_t)(uint32_t)vocab) >> 32);
  }
}

/* Raw bytes of a Q8_0-format tensor drawn directly (not by quantizing
 * anything): codes uniform in [-127, 127], scale bits = fp16 of a value drawn
 * uniformly in [lo, hi) (lo, hi > 0, both normal fp16 numbers), rounded by
 * truncating the mantissa to 10 bits.  Used to exercise the loader's Q8_0
 * input path with data that both sides receive byte for byte.
 * Layout per block: uint16 scale bits, then 32 int8 codes (34 bytes). */
void synth_q8_0_blocks(uint64_t seed, uint64_t stream, double lo, double hi,
                       int64_t nblocks, uint8_t* out) {
  const uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblocks; ++b) {
    uint8_t* blk = out + 34 * b;
    const uint64_t r0 = mix(key + 33 * (uint64_t)b);
    const double u = (double)(r0 >> 11) * (1.0 / 9007199254740992.0);
    const double v = lo + (hi - lo) * u;
    /* fp16 bits by truncation: v = m * 2^e with 1 <= m < 2 */
    int e = 0;
    double m = frexp(v, &e); /* v = m * 2^e, 0.5 <= m < 1 */
    m *= 2.0; e -= 1;
    const uint32_t mant = (uint32_t)((m - 1.0) * 1024.0); /* truncated */
    const uint16_t bits = (uint16_t)(((uint32_t)(e + 15) << 10) | mant);
    blk[0] = (uint8_t)(bits & 0xFF);
    blk[1] = (uint8_t)(bits >> 8);
    for (int k = 0; k < 32; ++k) {
      const uint64_t r = mix(key + 33 * (uint64_t)b + 1 + (uint64_t)k);
      const int code = (int)((r >> 32) % 255u) - 127;
      blk[2 + k] = (uint8_t)(int8_t)code;
    }
  }
}
