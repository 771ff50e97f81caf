/*
 * Seeded N(0, scale^2) bf16 inputs: the recipe of synthetic.py in C, threaded.
 *
 * Draw d of stream `seed` is splitmix64(seed + (d + 1) * 0x9E3779B97F4A7C15);
 * u = ((draw >> 11) + 1) * 2^-53 lies in (0, 1]; Box-Muller on draws (2p, 2p+1):
 * r = sqrt(-2 ln u1), x[2p] = r cos(2 pi u2), x[2p+1] = r sin(2 pi u2), in
 * double; then x * scale, rounded to float, then to bfloat16 (nearest even).
 * No attention arithmetic lives here.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

static uint64_t mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static uint16_t f32_to_bf16(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  return (uint16_t)((v.u + 0x7FFFu + ((v.u >> 16) & 1u)) >> 16);
}

typedef struct {
  uint64_t seed, p0, p1, count;
  double scale;
  uint16_t* out;
} Job;

static void* work(void* arg) {
  const Job* j = (const Job*)arg;
  for (uint64_t p = j->p0; p < j->p1; ++p) {
    const uint64_t z1 = mix(j->seed + (2 * p + 1) * 0x9E3779B97F4A7C15ull);
    const uint64_t z2 = mix(j->seed + (2 * p + 2) * 0x9E3779B97F4A7C15ull);
    const double u1 = ((double)(z1 >> 11) + 1.0) * (1.0 / 9007199254740992.0);
    const double u2 = ((double)(z2 >> 11) + 1.0) * (1.0 / 9007199254740992.0);
    const double r = sqrt(-2.0 * log(u1));
    const double a = 6.283185307179586 * u2;
    double x0 = r * cos(a), x1 = r * sin(a);
    if (j->scale != 1.0) {
      x0 = x0 * j->scale;
      x1 = x1 * j->scale;
    }
    j->out[2 * p] = f32_to_bf16((float)x0);
    if (2 * p + 1 < j->count) j->out[2 * p + 1] = f32_to_bf16((float)x1);
  }
  return NULL;
}

void synth_normal_bf16(uint64_t seed, uint64_t count, double scale, uint16_t* out, int nthreads) {
  const uint64_t npairs = (count + 1) / 2;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (npairs < 65536) nthreads = 1;
  pthread_t th[256];
  int created[256];
  Job jobs[256];
  const uint64_t per = (npairs + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].seed = seed;
    jobs[t].p0 = per * t < npairs ? per * t : npairs;
    jobs[t].p1 = per * (t + 1) < npairs ? per * (t + 1) : npairs;
    jobs[t].count = count;
    jobs[t].scale = scale;
    jobs[t].out = out;
    created[t] = t < nthreads - 1 && pthread_create(&th[t], NULL, work, &jobs[t]) == 0;
    if (!created[t]) work(&jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t)
    if (created[t]) pthread_join(th[t], NULL);
}
