/*
 * Seeded, counter-based synthetic input generator.
 *
 * This file holds no arithmetic of the attention method itself: it only
 * turns (stream key, element index) pairs into random numbers.  Both the
 * CUDA path's tests/benchmark and the CPU oracle's tests read the bytes it
 * writes, so the two sides always consume identical inputs.
 *
 * Definitions (all integer arithmetic is modulo 2^64):
 *   mix(z)        = SplitMix64 finaliser (Steele, Lea, Flood, "Fast
 *                   splittable pseudorandom number generators", OOPSLA 2014):
 *                   z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *                   z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31.
 *   draw(key, i)  = mix(key + (i + 1) * 0x9E3779B97F4A7C15), i.e. output i of
 *                   a SplitMix64 stream whose state starts at `key`.
 *   normal(key,i) = Box-Muller (cosine branch) on u1 = ((draw(key,2i) >> 11) + 1)
 *                   * 2^-53 in (0,1] and u2 = (draw(key,2i+1) >> 11) * 2^-53,
 *                   evaluated in fp64 with the C library's log/cos/sqrt.
 *   uniform_int(key, i, lo, hi): attempt r = 0,1,... draws
 *                   x = draw(key, i + r * 2^40) >> 32 and accepts the first
 *                   x < m * floor(2^32 / m) (m = hi - lo + 1); value = lo + x % m.
 *                   Exactly uniform; a rejection happens with probability < 4e-9.
 *
 * Every element depends only on (key, index), so any sub-range can be
 * generated on its own, and bulk ranges are split over POSIX threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

uint64_t csa2gen_stream_key(uint64_t config, uint64_t seed, uint64_t tensor) {
  uint64_t k = mix64(config * GOLDEN + 0x243F6A8885A308D3ULL);
  k = mix64(k ^ (seed * GOLDEN + 0x13198A2E03707344ULL));
  k = mix64(k ^ (tensor * GOLDEN + 0xA4093822299F31D0ULL));
  return k;
}

uint64_t csa2gen_draw(uint64_t key, uint64_t i) { return draw(key, i); }

static inline double normal_at(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  double u1 = (double)((draw(key, 2 * i) >> 11) + 1) * 0x1.0p-53;
  double u2 = (double)(draw(key, 2 * i + 1) >> 11) * 0x1.0p-53;
  return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

/* fp32 -> bf16 bits, round to nearest even (inputs are finite). */
static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static inline int32_t uniform_int_at(uint64_t key, uint64_t i, int32_t lo, int32_t hi) {
  uint64_t m = (uint64_t)(hi - lo) + 1;
  uint64_t lim = m * ((1ULL << 32) / m);
  for (uint64_t r = 0;; ++r) {
    uint64_t x = draw(key, i + (r << 40)) >> 32;
    if (x < lim) return lo + (int32_t)(x % m);
  }
}

enum { KIND_F64 = 0, KIND_F32 = 1, KIND_BF16 = 2, KIND_I8 = 3, KIND_I32 = 4 };

typedef struct {
  uint64_t key, start, count;
  int kind;
  int32_t lo, hi;
  void* out;
} job_t;

static void* run_job(void* p) {
  job_t* j = (job_t*)p;
  for (uint64_t t = 0; t < j->count; ++t) {
    uint64_t i = j->start + t;
    switch (j->kind) {
      case KIND_F64: ((double*)j->out)[t] = normal_at(j->key, i); break;
      case KIND_F32: ((float*)j->out)[t] = (float)normal_at(j->key, i); break;
      case KIND_BF16: ((uint16_t*)j->out)[t] = f32_to_bf16_rne((float)normal_at(j->key, i)); break;
      case KIND_I8: ((int8_t*)j->out)[t] = (int8_t)uniform_int_at(j->key, i, j->lo, j->hi); break;
      case KIND_I32: ((int32_t*)j->out)[t] = uniform_int_at(j->key, i, j->lo, j->hi); break;
    }
  }
  return 0;
}

static size_t elem_size(int kind) {
  switch (kind) {
    case KIND_F64: return 8;
    case KIND_F32: return 4;
    case KIND_BF16: return 2;
    case KIND_I8: return 1;
    default: return 4;
  }
}

static void run(uint64_t key, uint64_t start, uint64_t count, int kind, int32_t lo, int32_t hi,
                void* out, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (count < (1u << 16)) nthreads = 1;
  job_t jobs[64];
  pthread_t th[64];
  uint64_t per = (count + nthreads - 1) / nthreads;
  int launched = 0;
  for (int t = 0; t < nthreads; ++t) {
    uint64_t b = (uint64_t)t * per;
    if (b >= count) break;
    uint64_t e = b + per < count ? b + per : count;
    jobs[t].key = key;
    jobs[t].start = start + b;
    jobs[t].count = e - b;
    jobs[t].kind = kind;
    jobs[t].lo = lo;
    jobs[t].hi = hi;
    jobs[t].out = (char*)out + b * elem_size(kind);
    ++launched;
  }
  if (launched == 1) {
    run_job(&jobs[0]);
    return;
  }
  int started = 0;
  for (int t = 0; t < launched; ++t) {
    if (pthread_create(&th[t], 0, run_job, &jobs[t]) != 0) break;
    ++started;
  }
  for (int t = started; t < launched; ++t) run_job(&jobs[t]);
  for (int t = 0; t < started; ++t) pthread_join(th[t], 0);
}

void csa2gen_normal_f64(uint64_t key, uint64_t start, uint64_t count, double* out, int nthreads) {
  run(key, start, count, KIND_F64, 0, 0, out, nthreads);
}
void csa2gen_normal_f32(uint64_t key, uint64_t start, uint64_t count, float* out, int nthreads) {
  run(key, start, count, KIND_F32, 0, 0, out, nthreads);
}
void csa2gen_normal_bf16(uint64_t key, uint64_t start, uint64_t count, uint16_t* out, int nthreads) {
  run(key, start, count, KIND_BF16, 0, 0, out, nthreads);
}
void csa2gen_uniform_i8(uint64_t key, uint64_t start, uint64_t count, int32_t lo, int32_t hi,
                        int8_t* out, int nthreads) {
  run(key, start, count, KIND_I8, lo, hi, out, nthreads);
}
void csa2gen_uniform_i32(uint64_t key, uint64_t start, uint64_t count, int32_t lo, int32_t hi,
                         int32_t* out, int nthreads) {
  run(key, start, count, KIND_I32, lo, hi, out, nthreads);
}
