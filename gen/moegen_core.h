/*
 * Seeded synthetic-input generator: Philox4x32-10 counter-based integers and a
 * Box-Muller normal built only from IEEE-exact float operations (+ - * / sqrt).
 *
 * This header is the ONLY code shared between the CPU oracle side and the GPU
 * side of the project, and it holds none of the MoE layer's arithmetic: it
 * draws the random weights and activations that both sides consume.
 *
 * Determinism contract: every function here gives bit-identical results on the
 * host (gcc, -ffp-contract=off, no fast-math) and on the device (nvcc
 * -fmad=false, IEEE div/sqrt).  Nothing calls a libm or CUDA transcendental:
 * ln and cos are evaluated from their Taylor/atanh series with fixed constants
 * and a fixed operation order, so both compilers produce the same bits.
 *
 * Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 * as 1, 2, 3" (SC'11).  Round function, multipliers and Weyl key increments as
 * published there.
 *
 * Element addressing: element i of tensor (tensor_id, sub) under seed s uses
 * counter {lo32(i), hi32(i), tensor_id, sub} and key {lo32(s), hi32(s)}; word 0
 * gives u1 (radius), word 1 gives u2 (angle).  Any element can be drawn alone.
 */
#ifndef MOEGEN_CORE_H
#define MOEGEN_CORE_H

#include <stdint.h>

#ifdef __CUDACC__
#define MOEGEN_HD __host__ __device__ __forceinline__
#else
#define MOEGEN_HD static inline
#endif

#define MOEGEN_PHILOX_M0 0xD2511F53u
#define MOEGEN_PHILOX_M1 0xCD9E8D57u
#define MOEGEN_PHILOX_W0 0x9E3779B9u
#define MOEGEN_PHILOX_W1 0xBB67AE85u

MOEGEN_HD void moegen_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                                    uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k0 += MOEGEN_PHILOX_W0; k1 += MOEGEN_PHILOX_W1; }
    uint64_t p0 = (uint64_t)MOEGEN_PHILOX_M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)MOEGEN_PHILOX_M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

MOEGEN_HD int moegen_floor_log2_u32(uint32_t n) {  /* n >= 1 */
  int e = 0;
  while (n >> 1) { n >>= 1; ++e; }
  return e;
}

/* 2^e for integer e in [-126, 127], built from the exponent field (exact). */
MOEGEN_HD float moegen_pow2f(int e) {
  union { uint32_t u; float f; } v;
  v.u = (uint32_t)(e + 127) << 23;
  return v.f;
}

/*
 * ln(u) for u = (2a + 1) * 2^-24, a = r >> 9 (23 bits), so u lies in (0, 1).
 * u = m * 2^(e-24) with the odd integer n = 2a+1 = m * 2^e, m in (sqrt(2)/2, sqrt(2)].
 * ln m = 2 atanh(s), s = (m-1)/(m+1), |s| <= 0.1716, series to s^13.
 */
MOEGEN_HD float moegen_ln_u(uint32_t r) {
  const uint32_t n = 2u * (r >> 9) + 1u;        /* < 2^24: exact in float */
  int e = moegen_floor_log2_u32(n);
  float m = (float)n * moegen_pow2f(-e);        /* exact, in [1, 2) */
  if (m > 1.41421356f) { m = m * 0.5f; e = e + 1; }
  const float s = (m - 1.0f) / (m + 1.0f);
  const float s2 = s * s;
  float p = 1.0f / 13.0f;
  p = p * s2 + 1.0f / 11.0f;
  p = p * s2 + 1.0f / 9.0f;
  p = p * s2 + 1.0f / 7.0f;
  p = p * s2 + 1.0f / 5.0f;
  p = p * s2 + 1.0f / 3.0f;
  p = p * s2 + 1.0f;
  const float ln_m = 2.0f * s * p;
  const float ln2 = 0.693147180559945309f;
  return ln_m + (float)(e - 24) * ln2;
}

/*
 * cos(2 pi t) for t = q/4 + f/4, q = top two bits of r, f = (2b + 1) * 2^-23 with
 * b = bits 29..8 of r (22 bits), so f is exact in float and lies in (0, 1).
 * Quadrant symmetry reduces to an angle theta in [0, pi/4]; Taylor series
 * for cos to theta^12 and sin to theta^11.
 */
MOEGEN_HD float moegen_cos2pi_u(uint32_t r) {
  const uint32_t q = r >> 30;
  const uint32_t b = (r >> 8) & 0x3FFFFFu;
  float f = (float)(2u * b + 1u) * moegen_pow2f(-23);
  int swap = 0;
  if (f > 0.5f) { f = 1.0f - f; swap = 1; }       /* exact */
  const float half_pi = 1.57079632679489662f;
  const float th = f * half_pi;
  const float t2 = th * th;
  float c = 1.0f / 479001600.0f;                  /* 1/12! */
  c = c * (-t2) + 1.0f / 3628800.0f;              /* 1/10! */
  c = c * (-t2) + 1.0f / 40320.0f;                /* 1/8!  */
  c = c * (-t2) + 1.0f / 720.0f;                  /* 1/6!  */
  c = c * (-t2) + 1.0f / 24.0f;                   /* 1/4!  */
  c = c * (-t2) + 1.0f / 2.0f;                    /* 1/2!  */
  c = c * (-t2) + 1.0f;
  float s = 1.0f / 39916800.0f;                   /* 1/11! */
  s = s * (-t2) + 1.0f / 362880.0f;               /* 1/9!  */
  s = s * (-t2) + 1.0f / 5040.0f;                 /* 1/7!  */
  s = s * (-t2) + 1.0f / 120.0f;                  /* 1/5!  */
  s = s * (-t2) + 1.0f / 6.0f;                    /* 1/3!  */
  s = s * (-t2) + 1.0f;
  s = s * th;
  /* angle in quadrant = theta (or pi/2 - theta when swapped) */
  const float cq = swap ? s : c;   /* cos of the in-quadrant angle */
  const float sq = swap ? c : s;   /* sin of the in-quadrant angle */
  switch (q) {
    case 0: return cq;
    case 1: return -sq;
    case 2: return -cq;
    default: return sq;
  }
}

/* Standard normal draw for element i of (tensor, sub) under seed. */
MOEGEN_HD float moegen_std_normal(uint64_t seed, uint32_t tensor, uint32_t sub, uint64_t i) {
  const uint32_t ctr[4] = {(uint32_t)i, (uint32_t)(i >> 32), tensor, sub};
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t r[4];
  moegen_philox4x32_10(ctr, key, r);
  const float rad = -2.0f * moegen_ln_u(r[0]);
#ifdef __CUDA_ARCH__
  const float radius = __fsqrt_rn(rad);
#else
  const float radius = __builtin_sqrtf(rad);
#endif
  return radius * moegen_cos2pi_u(r[1]);
}

/* mean + std * z, with the two float operations kept separate. */
MOEGEN_HD float moegen_normal(uint64_t seed, uint32_t tensor, uint32_t sub, uint64_t i,
                              float mean, float stdev) {
  const float z = moegen_std_normal(seed, tensor, sub, i);
  const float t = stdev * z;
  return mean + t;
}

#endif /* MOEGEN_CORE_H */
