/*
 * Seeded synthetic input generator shared by the tests, the benchmark and the
 * oracle's callers.  It knows nothing about convolution: it only fills float
 * buffers with reproducible pseudo-random numbers.
 *
 * Element i of tensor t under seed s is derived from a counter-based hash
 * built on the SplitMix64 finaliser (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014):
 *
 *     mix(z)  = SplitMix64 output function applied to z + 0x9E3779B97F4A7C15
 *     h(s,t,i) = mix( mix(s) ^ (t * 0x9E3779B97F4A7C15) ^ i )
 *     u24      = h >> 40                      (top 24 bits)
 *     U[0,1)   = u24 * 2^-24                  (exact in float)
 *
 * Uniform ranges [lo, hi) are lo + (hi - lo) * U computed in double and
 * rounded once to float.  Normal samples use the Box-Muller transform in
 * double on the uniforms of counters 2i and 2i+1.  Because every element is a
 * pure function of (s, t, i), any element can be regenerated on its own and the
 * fill can be split across threads in any way without changing a bit.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z += GOLDEN;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t hash3(uint64_t seed, uint64_t tensor, uint64_t i) {
  return mix64(mix64(seed) ^ (tensor * GOLDEN) ^ i);
}

/* 24-bit uniform in [0,1). */
static inline double u01(uint64_t seed, uint64_t tensor, uint64_t i) {
  return (double)(hash3(seed, tensor, i) >> 40) * (1.0 / 16777216.0);
}

uint64_t synth_hash(uint64_t seed, uint64_t tensor, uint64_t i) { return hash3(seed, tensor, i); }

enum { KIND_UNIFORM = 0, KIND_NORMAL = 1 };

typedef struct {
  float *out;
  int64_t begin, end;
  uint64_t seed, tensor;
  double lo, hi;
  int kind;
} job_t;

static void *worker(void *arg) {
  job_t *j = (job_t *)arg;
  if (j->kind == KIND_UNIFORM) {
    const double span = j->hi - j->lo;
    for (int64_t i = j->begin; i < j->end; ++i)
      j->out[i] = (float)(j->lo + span * u01(j->seed, j->tensor, (uint64_t)i));
  } else {
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t i = j->begin; i < j->end; ++i) {
      /* u1 in (0,1] so that log(u1) is finite. */
      double u1 = ((double)(hash3(j->seed, j->tensor, 2 * (uint64_t)i) >> 40) + 1.0) * (1.0 / 16777216.0);
      double u2 = u01(j->seed, j->tensor, 2 * (uint64_t)i + 1);
      j->out[i] = (float)(sqrt(-2.0 * log(u1)) * cos(two_pi * u2));
    }
  }
  return NULL;
}

static int run(float *out, int64_t n, uint64_t seed, uint64_t tensor, double lo, double hi, int kind,
               int nthreads) {
  if (!out || n < 0) return 1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < 65536) nthreads = 1;
  pthread_t tid[256];
  job_t jobs[256];
  int64_t chunk = (n + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    int64_t b = t * chunk, e = b + chunk;
    if (b > n) b = n;
    if (e > n) e = n;
    jobs[t] = (job_t){out, b, e, seed, tensor, lo, hi, kind};
    if (t == nthreads - 1 || pthread_create(&tid[t], NULL, worker, &jobs[t]) != 0) {
      worker(&jobs[t]);
    } else {
      started = t + 1;
    }
  }
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  return 0;
}

/* out[i] = lo + (hi-lo)*U_i, i in [0, n). Returns 0 on success. */
int synth_uniform_f32(float *out, int64_t n, uint64_t seed, uint64_t tensor, double lo, double hi,
                      int nthreads) {
  return run(out, n, seed, tensor, lo, hi, KIND_UNIFORM, nthreads);
}

/* out[i] ~ N(0,1) by Box-Muller on counters (2i, 2i+1). Returns 0 on success. */
int synth_normal_f32(float *out, int64_t n, uint64_t seed, uint64_t tensor, int nthreads) {
  return run(out, n, seed, tensor, 0.0, 0.0, KIND_NORMAL, nthreads);
}

/* Regenerate selected elements (by flat index) without filling the whole tensor. */
int synth_uniform_at(float *out, const int64_t *idx, int64_t n, uint64_t seed, uint64_t tensor, double lo,
                     double hi) {
  if (!out || !idx || n < 0) return 1;
  for (int64_t k = 0; k < n; ++k)
    out[k] = (float)(lo + (hi - lo) * u01(seed, tensor, (uint64_t)idx[k]));
  return 0;
}
