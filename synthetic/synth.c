/*
 * Seeded, position-addressable synthetic inputs shared by the oracle-side
 * tests and the GPU-side tests/benchmark.
 *
 * This file holds no arithmetic of the compressor itself: it only draws
 * numbers.  Every value is a pure function of (seed, tensor id, stream,
 * index), so any element (for example token t of sequence b) can be
 * regenerated on its own, independent of how much else is generated.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  Element i of a stream
 * keyed by k is the SplitMix64 output after i+1 increments of the state
 * starting at k.  The stream key is itself a SplitMix64 mix of the seed,
 * tensor id and stream number.
 *
 * Uniform: the top 53 bits of an output, scaled to [0, 1).
 * Normal:  Box-Muller on the uniforms of indices (2i, 2i+1) of the same
 *          stream, computed in double and rounded once to float.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define SM_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid, uint64_t stream) {
  uint64_t a = sm_mix(tid * 0xD1B54A32D192ED03ULL + stream + SM_GAMMA);
  return sm_mix(seed * SM_GAMMA ^ a);
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return sm_mix(key + (i + 1) * SM_GAMMA); }

static inline double unif(uint64_t key, uint64_t i) {
  return (double)(draw(key, i) >> 11) * (1.0 / 9007199254740992.0);
}

static inline double normal(uint64_t key, uint64_t i) {
  double u1 = 1.0 - unif(key, 2 * i); /* (0, 1] */
  double u2 = unif(key, 2 * i + 1);
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* ---- threaded fill ------------------------------------------------------ */

typedef struct {
  uint64_t key;
  uint64_t first; /* index of out[0] within the stream */
  int64_t lo, hi; /* range of out handled by this thread */
  double mean, scale;
  float* out;
  int kind; /* 0 normal, 1 uniform */
} fill_job;

static void* fill_worker(void* p) {
  fill_job* j = (fill_job*)p;
  for (int64_t i = j->lo; i < j->hi; ++i) {
    double v = j->kind == 0 ? normal(j->key, j->first + (uint64_t)i) : unif(j->key, j->first + (uint64_t)i);
    j->out[i] = (float)(j->mean + j->scale * v);
  }
  return NULL;
}

static void fill(uint64_t key, uint64_t first, int64_t count, double mean, double scale, float* out, int kind,
                 int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (count < (int64_t)1 << 16) nthreads = 1;
  pthread_t th[64];
  fill_job jobs[64];
  int64_t per = (count + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].key = key;
    jobs[t].first = first;
    jobs[t].lo = (int64_t)t * per;
    jobs[t].hi = jobs[t].lo + per < count ? jobs[t].lo + per : count;
    jobs[t].mean = mean;
    jobs[t].scale = scale;
    jobs[t].out = out;
    jobs[t].kind = kind;
    if (jobs[t].lo >= jobs[t].hi) break;
    if (t == 0) continue;
    if (pthread_create(&th[t], NULL, fill_worker, &jobs[t]) != 0) {
      fill_worker(&jobs[t]); /* run inline if a thread cannot be started */
      jobs[t].lo = jobs[t].hi;
      th[t] = 0;
    }
    started = t + 1;
  }
  fill_worker(&jobs[0]);
  for (int t = 1; t < started; ++t)
    if (th[t]) pthread_join(th[t], NULL);
}

/* out[i] = mean + scale * N(0,1) at stream indices first..first+count-1 */
void synth_normal(uint64_t seed, uint64_t tid, uint64_t stream, uint64_t first, int64_t count, double mean,
                  double scale, float* out, int nthreads) {
  fill(stream_key(seed, tid, stream), first, count, mean, scale, out, 0, nthreads);
}

/* out[i] = U[0,1) at stream indices first..first+count-1 */
void synth_uniform(uint64_t seed, uint64_t tid, uint64_t stream, uint64_t first, int64_t count, float* out,
                   int nthreads) {
  fill(stream_key(seed, tid, stream), first, count, 0.0, 1.0, out, 1, nthreads);
}

/* one uniform in double, for decisions (outlier masks, start positions) */
double synth_uniform1(uint64_t seed, uint64_t tid, uint64_t stream, uint64_t index) {
  return unif(stream_key(seed, tid, stream), index);
}
