/*
 * Seeded synthetic inputs for the routed MoE layer.
 *
 * This file holds no step of the layer itself: it only draws numbers.
 * Both the CPU oracle (via the tests) and the CUDA path (via the tests,
 * smoke() and bench.py) take their inputs from here.
 *
 * Generator: a counter-based stream.  Element n of stream `stream` under
 * `seed` is built from two 64-bit words
 *     w(c) = mix64(key + (c + 1) * 0x9E3779B97F4A7C15),  c = 2*(n/2), 2*(n/2)+1
 * with key = mix64(seed * 0xD1B54A32D192ED03 + stream) and mix64 the
 * SplitMix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014).  The two words give two uniforms in
 * (0, 1] and a Box-Muller pair (Box & Muller 1958); even n takes the
 * cosine branch and odd n the sine branch.  Every element depends only on
 * (seed, stream, n), so the fill is identical for any thread count and on
 * any machine.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * 0xD1B54A32D192ED03ull + stream);
}

static inline double unit_open0(uint64_t key, uint64_t c) {
  uint64_t w = mix64(key + (c + 1ull) * 0x9E3779B97F4A7C15ull);
  return ((double)(w >> 11) + 1.0) * (1.0 / 9007199254740992.0); /* (0, 1] */
}

static inline double normal_at(uint64_t key, uint64_t n) {
  uint64_t pair = n >> 1;
  double u1 = unit_open0(key, 2 * pair);
  double u2 = unit_open0(key, 2 * pair + 1);
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  return (n & 1) ? r * sin(th) : r * cos(th);
}

/* fp32 -> bf16 bits, round to nearest even (inputs here are finite). */
static inline uint16_t to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

typedef struct {
  uint16_t *out;
  size_t begin, end;
  uint64_t key;
  double sigma;
} normal_job;

static void *normal_worker(void *arg) {
  normal_job *j = (normal_job *)arg;
  for (size_t n = j->begin; n < j->end; ++n)
    j->out[n] = to_bf16_bits((float)(normal_at(j->key, n) * j->sigma));
  return NULL;
}

/* out[n] = bf16(float(sigma * N(0,1)_n)), n in [0, count). */
void synth_normal_bf16(uint16_t *out, size_t count, uint64_t seed,
                       uint64_t stream, double sigma, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((size_t)nthreads > count / 65536 + 1) nthreads = (int)(count / 65536 + 1);
  pthread_t th[256];
  normal_job jobs[256];
  uint64_t key = stream_key(seed, stream);
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].out = out;
    jobs[i].begin = count * (size_t)i / (size_t)nthreads;
    jobs[i].end = count * (size_t)(i + 1) / (size_t)nthreads;
    jobs[i].key = key;
    jobs[i].sigma = sigma;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, normal_worker, &jobs[i]);
  normal_worker(&jobs[0]);
  for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* A seeded permutation of 0..n-1 (Fisher-Yates, Durstenfeld form). */
void synth_permutation(int32_t *perm, int n, uint64_t seed, uint64_t stream) {
  uint64_t key = stream_key(seed, stream);
  for (int i = 0; i < n; ++i) perm[i] = i;
  for (int i = n - 1; i > 0; --i) {
    uint64_t w = mix64(key + ((uint64_t)i + 1ull) * 0x9E3779B97F4A7C15ull);
    int j = (int)(w % (uint64_t)(i + 1));
    int32_t t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
}

static inline double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

typedef struct {
  const uint16_t *x, *wr;
  const double *bias;
  float *logits;
  int t0, t1, H, E;
} logit_job;

static void *logit_worker(void *arg) {
  logit_job *j = (logit_job *)arg;
  for (int t = j->t0; t < j->t1; ++t) {
    const uint16_t *xr = j->x + (size_t)t * j->H;
    for (int e = 0; e < j->E; ++e) {
      const uint16_t *wrow = j->wr + (size_t)e * j->H;
      double acc = 0.0;
      for (int h = 0; h < j->H; ++h) acc += bf16_value(xr[h]) * bf16_value(wrow[h]);
      if (j->bias) acc += j->bias[e];
      j->logits[(size_t)t * j->E + e] = (float)acc;
    }
  }
  return NULL;
}

/*
 * Router logits handed to the layer as its input:
 *   logits[t,e] = float( sum_h x[t,h] * Wr[e,h]  + bias[e] )
 * summed in double, h ascending, rounded to float once.  (The projection
 * that produces logits is upstream of the routed layer; it is evaluated
 * here only to give the logits the scale and correlations of a real router.)
 */
void synth_router_logits(const uint16_t *x, const uint16_t *wr, const double *bias,
                         int T, int H, int E, float *logits, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > T) nthreads = T > 0 ? T : 1;
  pthread_t th[256];
  logit_job jobs[256];
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].x = x;
    jobs[i].wr = wr;
    jobs[i].bias = bias;
    jobs[i].logits = logits;
    jobs[i].t0 = (int)((long long)T * i / nthreads);
    jobs[i].t1 = (int)((long long)T * (i + 1) / nthreads);
    jobs[i].H = H;
    jobs[i].E = E;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, logit_worker, &jobs[i]);
  logit_worker(&jobs[0]);
  for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
}
