/*
 * Host side of the seeded synthetic-input generator (see moegen_core.h).
 * Compiled with -ffp-contract=off so the float arithmetic is bit-identical to
 * the device kernel in moegen_cuda.cu.  Exposed through ctypes.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include "moegen_core.h"

void moegen_philox(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  moegen_philox4x32_10(ctr, key, out);
}

float moegen_ln_u_host(uint32_t r) { return moegen_ln_u(r); }
float moegen_cos2pi_u_host(uint32_t r) { return moegen_cos2pi_u(r); }

typedef struct {
  uint64_t seed; uint32_t tensor, sub; uint64_t start, n; float mean, stdev; float* out;
} job_t;

static void* run_job(void* p) {
  job_t* j = (job_t*)p;
  for (uint64_t t = 0; t < j->n; ++t)
    j->out[t] = moegen_normal(j->seed, j->tensor, j->sub, j->start + t, j->mean, j->stdev);
  return NULL;
}

/* out[t] = normal draw of element (start + t), t in [0, n).  nthreads >= 1. */
void moegen_normal_f32(uint64_t seed, uint32_t tensor, uint32_t sub, uint64_t start, uint64_t n,
                       float mean, float stdev, float* out, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if ((uint64_t)nthreads > n / 65536 + 1) nthreads = (int)(n / 65536 + 1);
  job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nthreads);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  uint64_t per = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
  for (int i = 0; i < nthreads; ++i) {
    uint64_t a = per * (uint64_t)i, b = a + per;
    if (a > n) a = n;
    if (b > n) b = n;
    jobs[i] = (job_t){seed, tensor, sub, start + a, b - a, mean, stdev, out + a};
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, run_job, &jobs[i]);
  run_job(&jobs[0]);
  for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
  free(jobs);
  free(th);
}
