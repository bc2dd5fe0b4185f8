/* Seeded synthetic inputs for the hyper-connection read.
 *
 * This module only draws random numbers; it holds none of the read's
 * arithmetic.  Both the CUDA path's tests/benchmark and the FP64 oracle take
 * their inputs from it, so the two sides see the same bytes.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used in counter form: draw j of a stream
 * with key k is mix(k + (j + 1) * gamma), so any element can be produced
 * independently and the output does not depend on the number of threads.
 * Normal deviates come from the Box-Muller transform (Box and Muller, 1958):
 * draws 2p and 2p+1 give the pair (r cos(2 pi u2), r sin(2 pi u2)) with
 * r = sqrt(-2 ln u1).  BF16 values are the binary32 draw rounded to nearest,
 * ties to even, on its upper 16 bits.
 *
 * Build with -ffp-contract=off so that aarch64 and x86-64 hosts agree.
 */

#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define HC_GAMMA 0x9e3779b97f4a7c15ULL

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

/* Key of the stream for tensor `tensor_id` under seed `seed`. */
static uint64_t stream_key(uint64_t seed, uint32_t tensor_id) {
  return mix64(mix64(seed) ^ ((uint64_t)(tensor_id + 1) * HC_GAMMA));
}

static uint64_t draw(uint64_t key, uint64_t j) { return mix64(key + (j + 1) * HC_GAMMA); }

/* Normal deviate number `idx` of the stream (mean 0, variance 1). */
static double normal_at(uint64_t key, uint64_t idx) {
  const uint64_t p = idx >> 1;
  const double two_pi = 6.283185307179586476925286766559;
  const double u1 = (double)((draw(key, 2 * p) >> 11) + 1) * 0x1.0p-53; /* (0, 1] */
  const double u2 = (double)(draw(key, 2 * p + 1) >> 11) * 0x1.0p-53;   /* [0, 1) */
  const double r = sqrt(-2.0 * log(u1));
  return (idx & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

typedef struct {
  uint64_t key;
  double mean, std;
  size_t begin, end;
  float* f32;
  uint16_t* bf16;
} job_t;

static void* run_job(void* arg) {
  job_t* j = (job_t*)arg;
  for (size_t i = j->begin; i < j->end; ++i) {
    float v = (float)(j->mean + j->std * normal_at(j->key, i));
    if (j->f32) j->f32[i] = v;
    else j->bf16[i] = f32_to_bf16_rne(v);
  }
  return NULL;
}

static void fill(uint64_t seed, uint32_t tensor_id, double mean, double std, float* f32,
                 uint16_t* bf16, size_t n, int threads) {
  enum { MAXT = 64 };
  pthread_t tid[MAXT];
  int joined[MAXT];
  job_t jobs[MAXT];
  const uint64_t key = stream_key(seed, tensor_id);
  if (threads < 1) threads = 1;
  if (threads > MAXT) threads = MAXT;
  if (n < (size_t)1 << 16) threads = 1;
  const size_t chunk = (n + (size_t)threads - 1) / (size_t)threads;
  for (int t = 0; t < threads; ++t) {
    size_t b = (size_t)t * chunk, e = b + chunk;
    if (b > n) b = n;
    if (e > n) e = n;
    jobs[t] = (job_t){key, mean, std, b, e, f32, bf16};
    joined[t] = 0;
    if (t == 0) continue;
    if (pthread_create(&tid[t], NULL, run_job, &jobs[t]) == 0) {
      joined[t] = 1;
    } else {
      run_job(&jobs[t]); /* no thread available: do the chunk here */
    }
  }
  run_job(&jobs[0]);
  for (int t = 1; t < threads; ++t) {
    if (joined[t]) pthread_join(tid[t], NULL);
  }
}

/* out[i] = float(mean + std * z_i), z_i the i-th normal deviate of the stream. */
void hc_synth_normal_f32(uint64_t seed, uint32_t tensor_id, double mean, double std,
                         float* out, size_t n, int threads) {
  fill(seed, tensor_id, mean, std, out, NULL, n, threads);
}

/* out[i] = bf16_rne(float(mean + std * z_i)). */
void hc_synth_normal_bf16(uint64_t seed, uint32_t tensor_id, double mean, double std,
                          uint16_t* out, size_t n, int threads) {
  fill(seed, tensor_id, mean, std, NULL, out, n, threads);
}

/* Raw draw j of a stream, exposed so tests can check the generator against
 * published SplitMix64 output. */
uint64_t hc_synth_raw(uint64_t key, uint64_t j) { return draw(key, j); }
uint64_t hc_synth_mix64(uint64_t z) { return mix64(z); }
