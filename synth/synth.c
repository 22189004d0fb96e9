/*
 * synth.c -- seeded, counter-based synthetic inputs shared by the oracle
 * tests and the CUDA path.
 *
 * This module holds no arithmetic of the decoder: it only turns
 * (seed, tensor id, element index) into numbers.  Every element depends on
 * those three values alone, so results do not depend on the thread count or
 * on the machine (x86_64 here, aarch64 on the GPU host).
 *
 * Generator (published definitions, restated):
 *   splitmix64(x): z = x + 0x9E3779B97F4A7C15; z = (z ^ z>>30) * 0xBF58476D1CE4E5B9;
 *                  z = (z ^ z>>27) * 0x94D049BB133111EB; return z ^ z>>31.
 *   (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
 *    OOPSLA 2014; the mixing constants are Stafford's variant 13.)
 *   key(seed, t, i) = seed ^ (t << 40) ^ i
 *   normal(seed, t, i): z1 = splitmix64(key(seed,t,2i)), z2 = splitmix64(key(seed,t,2i+1));
 *       u1 = ((z1 >> 11) + 1) * 2^-53 in (0,1], u2 = (z2 >> 11) * 2^-53 in [0,1);
 *       n = sqrt(-2 ln u1) * cos(2 pi u2)                      (Box-Muller, 1958)
 *   bf16 value: v = (float)(mean + std * n), then round-to-nearest-even to bf16.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

static inline uint64_t sm64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t key_of(uint64_t seed, uint32_t tid, uint64_t i) {
  return seed ^ ((uint64_t)tid << 40) ^ i;
}

static inline double normal_at(uint64_t seed, uint32_t tid, uint64_t i) {
  uint64_t z1 = sm64(key_of(seed, tid, 2 * i));
  uint64_t z2 = sm64(key_of(seed, tid, 2 * i + 1));
  double u1 = ((double)(z1 >> 11) + 1.0) * 0x1.0p-53;
  double u2 = (double)(z2 >> 11) * 0x1.0p-53;
  return sqrt(-2.0 * log(u1)) * cos(2.0 * M_PI * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

uint64_t synth_splitmix64(uint64_t x) { return sm64(x); }

double synth_normal(uint64_t seed, uint32_t tid, uint64_t i) {
  return normal_at(seed, tid, i);
}

uint16_t synth_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }

/* ---- multi-threaded fills ------------------------------------------------ */

typedef struct {
  int kind; /* 0: normal bf16, 1: kv prefill */
  uint64_t seed;
  uint32_t tid;
  uint64_t lo, hi; /* element range [lo, hi) */
  double mean, std;
  uint16_t *out;
  /* kv prefill geometry */
  int64_t nkv, max_ctx, d, batch;
  const int32_t *ctx;
} job_t;

static void *run_job(void *arg) {
  job_t *j = (job_t *)arg;
  if (j->kind == 0) {
    for (uint64_t i = j->lo; i < j->hi; ++i)
      j->out[i] = f32_to_bf16_rne((float)(j->mean + j->std * normal_at(j->seed, j->tid, i)));
  } else {
    /* tensor [L][B][nkv][max_ctx][d]; positions p < ctx[b] hold N(mean,std), others 0 */
    for (uint64_t i = j->lo; i < j->hi; ++i) {
      uint64_t p = (i / (uint64_t)j->d) % (uint64_t)j->max_ctx;
      uint64_t b = (i / ((uint64_t)j->d * j->max_ctx * j->nkv)) % (uint64_t)j->batch;
      if ((int64_t)p < (int64_t)j->ctx[b])
        j->out[i] = f32_to_bf16_rne((float)(j->mean + j->std * normal_at(j->seed, j->tid, i)));
      else
        j->out[i] = 0;
    }
  }
  return 0;
}

static void run_parallel(job_t proto, uint64_t n, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > n / 65536 + 1) nthreads = (int)(n / 65536 + 1);
  pthread_t th[256];
  int threaded[256];
  job_t jobs[256];
  uint64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].lo = (uint64_t)t * per;
    if (jobs[t].lo > n) jobs[t].lo = n;
    jobs[t].hi = jobs[t].lo + per > n ? n : jobs[t].lo + per;
    threaded[t] = 0;
    if (t > 0 && jobs[t].lo < jobs[t].hi) {
      if (pthread_create(&th[t], 0, run_job, &jobs[t]) == 0)
        threaded[t] = 1;
      else
        run_job(&jobs[t]);
    }
  }
  if (n > 0) run_job(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (threaded[t]) pthread_join(th[t], 0);
}

/* out[i] = bf16(mean + std * normal(seed, tid, i)), i in [0, n) */
void synth_normal_bf16(uint64_t seed, uint32_t tid, uint64_t n, double mean, double std,
                       uint16_t *out, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = 0;
  j.seed = seed;
  j.tid = tid;
  j.mean = mean;
  j.std = std;
  j.out = out;
  run_parallel(j, n, nthreads);
}

/* KV-cache prefill for a [L][B][nkv][max_ctx][d] bf16 tensor: N(mean,std) at
   positions p < ctx[b], zero elsewhere. */
void synth_kv_bf16(uint64_t seed, uint32_t tid, int64_t L, int64_t B, int64_t nkv,
                   int64_t max_ctx, int64_t d, const int32_t *ctx, double mean, double std,
                   uint16_t *out, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = 1;
  j.seed = seed;
  j.tid = tid;
  j.mean = mean;
  j.std = std;
  j.out = out;
  j.nkv = nkv;
  j.max_ctx = max_ctx;
  j.d = d;
  j.batch = B;
  j.ctx = ctx;
  run_parallel(j, (uint64_t)(L * B * nkv * max_ctx * d), nthreads);
}

/* out[i] = lo + splitmix64(key(seed, tid, i)) mod (hi - lo + 1), inclusive range */
void synth_uniform_i32(uint64_t seed, uint32_t tid, uint64_t n, int64_t lo, int64_t hi,
                       int32_t *out) {
  uint64_t span = (uint64_t)(hi - lo + 1);
  for (uint64_t i = 0; i < n; ++i) out[i] = (int32_t)(lo + (int64_t)(sm64(key_of(seed, tid, i)) % span));
}
