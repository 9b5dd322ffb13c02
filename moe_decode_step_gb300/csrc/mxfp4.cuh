// MXFP4 packing (host and device) and the debug dequantiser.
//
// Encoding (OCP Microscaling Formats (MX) v1.0): E2M1 elements, one E8M0 scale
// per 32 contiguous K elements.  Scale exponent = floor(log2 amax) - 2,
// clamped to [-127, 127] (an all-zero block takes -127), so amax / 2^e lies in
// [4, 8).  Each element w / 2^e (exact: a power-of-two scaling) is rounded to
// the E2M1 grid {0, .5, 1, 1.5, 2, 3, 4, 6} to nearest, ties to the even code,
// saturating at 6; the sign bit is the sign of w.  Canonical layout: byte j of
// a row holds elements 2j (low nibble) and 2j + 1 (high nibble).
#pragma once

#include <math.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"

namespace moe {

// floor(log2 |v|) of a finite non-zero float from its bit pattern.
__host__ __device__ inline int floor_log2_bits(uint32_t bits) {
  const uint32_t ex = (bits >> 23) & 0xFF;
  if (ex != 0) return (int)ex - 127;
  const uint32_t man = bits & 0x7FFFFF;   // subnormal: value = man * 2^-149
  int msb = 31;
  while (!(man >> msb & 1u)) --msb;
  return msb - 149;
}

__host__ __device__ inline int mx_block_exponent(float amax) {
  if (amax == 0.0f) return -127;
  uint32_t bits;
  memcpy(&bits, &amax, 4);
  int e = floor_log2_bits(bits) - 2;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Nearest E2M1 magnitude code for a >= 0; the midpoints 0.25, 1.25, 2.5, 5
// round down (to the even codes 0, 2, 4, 6) and 0.75, 1.75, 3.5 round up (to
// the even codes 2, 4, 6).  Values above 5 become 6 (code 7), which also
// saturates everything larger.
__host__ __device__ inline uint32_t e2m1_magnitude_code(float a) {
  return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
         (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
         (uint32_t)(a > 5.0f);
}

// Pack one 32-element block: 16 nibble bytes and the scale byte.
__host__ __device__ inline uint8_t mx_pack_block(const float* w, uint8_t* q16) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(w[i]));
  const int e = mx_block_exponent(amax);
  for (int i = 0; i < 32; i += 2) {
    uint32_t c[2];
    for (int t = 0; t < 2; ++t) {
      const float v = ldexpf(w[i + t], -e);   // exact power-of-two scaling
      uint32_t bits;
      memcpy(&bits, &v, 4);
      c[t] = (bits >> 28 & 8u) | e2m1_magnitude_code(fabsf(v));
    }
    q16[i / 2] = (uint8_t)(c[0] | c[1] << 4);
  }
  return (uint8_t)(e + 127);
}

__global__ void mxfp4_pack_kernel(const float* __restrict__ w, int64_t rows, int64_t k,
                                  uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  const int64_t nb = k / 32;
  const int64_t total = rows * nb;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / nb, b = t % nb;
    float blk[32];
    const float4* src = reinterpret_cast<const float4*>(w + r * k + b * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = src[i];
      blk[4 * i] = v.x;
      blk[4 * i + 1] = v.y;
      blk[4 * i + 2] = v.z;
      blk[4 * i + 3] = v.w;
    }
    uint8_t qb[16];
    s[r * nb + b] = mx_pack_block(blk, qb);
    uint4 out;
    memcpy(&out, qb, 16);
    *reinterpret_cast<uint4*>(q + r * (k / 2) + b * 16) = out;
  }
}

// Dequantise rows x k through the GEMV kernels' decode path
// (cvt.rn.f16x2.e2m1x2 and the E8M0 scale) into fp32.
__global__ void mxfp4_dequant_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                     int64_t rows, int64_t k, float* __restrict__ out) {
  const int64_t nb = k / 32;
  const int64_t total = rows * nb;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / nb, b = t % nb;
    const uint4 v = *reinterpret_cast<const uint4*>(q + r * (k / 2) + b * 16);
    const float sc = e8m0_to_f32(s[r * nb + b]);
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    float* o = out + r * k + b * 32;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t hq[4];
      e2m1x8_to_f16x2(words[w], hq);
#pragma unroll
      for (int t2 = 0; t2 < 4; ++t2) {
        o[w * 8 + t2 * 2 + 0] = f16_lo(hq[t2]) * sc;
        o[w * 8 + t2 * 2 + 1] = f16_hi(hq[t2]) * sc;
      }
    }
  }
}

}  // namespace moe
