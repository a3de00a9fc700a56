/*
 * Seeded synthetic input generator shared by the CUDA path's tests/bench and
 * the CPU oracle's tests.  It holds none of the attention arithmetic: it only
 * turns (seed, stream, index) into numbers.
 *
 *  - counter-based splitmix64 (Steele, Lea, Flood, "Fast splittable
 *    pseudorandom number generators", OOPSLA 2014; constants as published by
 *    Vigna) -> 53-bit uniforms;
 *  - Box-Muller transform (Box & Muller, 1958) -> standard normals in double,
 *    rounded once to fp32, multiplied by a fp32 factor, then (optionally)
 *    rounded to bf16 with round-to-nearest-even;
 *  - bounded integers with Lemire's multiply-shift + rejection method
 *    (Lemire, "Fast random integer generation in an interval", 2019).
 *
 * Element i of stream s under seed S depends only on (S, s, i), so any slice
 * can be produced independently and by any number of threads.  Plain C99 +
 * pthreads, no architecture-specific code (it runs on x86_64 and aarch64).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static uint64_t sm64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Per-(seed, stream) key; the counter for draw c is key + c (golden-ratio
 * increments happen inside sm64, so consecutive counters are decorrelated). */
static uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return sm64(sm64(seed) ^ (stream * 0xD1B54A32D192ED03ULL));
}

static double u53_open0(uint64_t x) { /* (0, 1] */
  return ((double)(x >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}
static double u53(uint64_t x) { /* [0, 1) */
  return (double)(x >> 11) * (1.0 / 9007199254740992.0);
}

/* Standard normal number i of the stream (pair p = i/2 uses draws 2p, 2p+1). */
static double normal_at(uint64_t key, int64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t p = (uint64_t)i >> 1;
  double u1 = u53_open0(sm64(key + 2 * p));
  double u2 = u53(sm64(key + 2 * p + 1));
  double r = sqrt(-2.0 * log(u1));
  return (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return 0x7FC0; /* NaN */
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7FFFu + lsb;
  return (uint16_t)(b >> 16);
}

typedef struct {
  uint64_t key;
  float mult;
  int kind; /* 0 = bf16 bits, 1 = fp32 */
  void *out;
  int64_t lo, hi;
} job_t;

static void *run_job(void *arg) {
  job_t *j = (job_t *)arg;
  for (int64_t i = j->lo; i < j->hi; ++i) {
    float f = (float)normal_at(j->key, i);
    f = f * j->mult;
    if (j->kind == 0)
      ((uint16_t *)j->out)[i] = f32_to_bf16_rne(f);
    else
      ((float *)j->out)[i] = f;
  }
  return 0;
}

static void fill(uint64_t seed, uint64_t stream, float mult, int kind, void *out, int64_t n,
                 int nthreads) {
  if (n <= 0) return;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < (int64_t)1 << 16) nthreads = 1;
  pthread_t th[256];
  job_t jobs[256];
  uint64_t key = stream_key(seed, stream);
  int64_t chunk = (n + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].key = key;
    jobs[t].mult = mult;
    jobs[t].kind = kind;
    jobs[t].out = out;
    jobs[t].lo = (int64_t)t * chunk;
    jobs[t].hi = jobs[t].lo + chunk < n ? jobs[t].lo + chunk : n;
    if (jobs[t].lo >= jobs[t].hi) break;
    if (t == 0) continue;
    if (pthread_create(&th[t], 0, run_job, &jobs[t]) != 0) {
      run_job(&jobs[t]);
      jobs[t].hi = jobs[t].lo; /* mark as done inline */
      th[t] = 0;
    }
    started = t;
  }
  run_job(&jobs[0]);
  for (int t = 1; t <= started; ++t)
    if (jobs[t].hi > jobs[t].lo) pthread_join(th[t], 0);
}

/* n normals x mult, each rounded to fp32 then (after the fp32 multiply) to bf16. */
void ig_normal_bf16(uint64_t seed, uint64_t stream, float mult, uint16_t *out, int64_t n,
                    int nthreads) {
  fill(seed, stream, mult, 0, out, n, nthreads);
}

/* n normals x sigma as fp32. */
void ig_normal_f32(uint64_t seed, uint64_t stream, float sigma, float *out, int64_t n,
                   int nthreads) {
  fill(seed, stream, sigma, 1, out, n, nthreads);
}

/* n integers uniform in [lo, hi] (inclusive), unbiased (Lemire with rejection). */
int ig_uniform_int(uint64_t seed, uint64_t stream, int32_t lo, int32_t hi, int32_t *out,
                   int64_t n) {
  if (hi < lo) return -1;
  uint64_t key = stream_key(seed, stream);
  uint64_t range = (uint64_t)((int64_t)hi - (int64_t)lo) + 1u; /* <= 2^32 */
  uint64_t ctr = 0;
  for (int64_t i = 0; i < n; ++i) {
    if (range == (uint64_t)1 << 32) {
      out[i] = (int32_t)((int64_t)lo + (int64_t)(sm64(key + ctr++) >> 32));
      continue;
    }
    uint32_t r32 = (uint32_t)range;
    uint64_t m = (sm64(key + ctr++) >> 32) * (uint64_t)r32;
    uint32_t l = (uint32_t)m;
    if (l < r32) {
      uint32_t t = (uint32_t)(-r32) % r32;
      while (l < t) {
        m = (sm64(key + ctr++) >> 32) * (uint64_t)r32;
        l = (uint32_t)m;
      }
    }
    out[i] = (int32_t)((int64_t)lo + (int64_t)(m >> 32));
  }
  return 0;
}
