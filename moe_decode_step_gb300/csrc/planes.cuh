// Activation planes: the activation operand of the block-scaled tensor-core
// expert matmuls (E2M1 weights x E2M1 activations, E8M0 scales per 32 K).
//
// A row v of K activations becomes 8 E2M1 planes q_0..q_7 with scales s_p =
// 2^(c - 127 - 2p), v = sum_p s_p q_p + r.  c is the smallest power of two
// with 6 * 2^(c-127) >= max|v| over the set it covers (one code per
// 32-element block, or one per row), so plane 0 never saturates.  Each plane rounds the running residual to the
// E2M1 grid; the widest grid gap (4 -> 6) bounds that rounding error by s_p =
// 4 s_{p+1}, so the next plane's input again lies within +-4 of its grid and
// never saturates either.  After 8 planes |r| <= s_7 = 2^-14 s_0, below
// max|v| * 2^-14 / 3 per element (max over the code's block or row): products with the exact E2M1 weights then
// sum on the tensor cores in fp32 with an error far below the fp32 rounding
// of the sums themselves.  (A plane's code is clamped at 1, the smallest
// normal E8M0 scale; a clamped plane repeats the previous scale, which keeps
// its input in range.)
//
// Storage of one row (K elements): 128 bytes per 32-element block b, at
// b * 128: plane p's 16 bytes at + p * 16, element 2j in the low nibble of
// byte j and element 2j + 1 in the high nibble.  So the 8 planes of one block
// form one 8-row x 16-byte core matrix of the tensor-core B operand, and any
// run of blocks is contiguous.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace moe {

constexpr int kPlanes = 8;

// Bytes of a row's planes / codes.
__host__ __device__ inline size_t planes_row_bytes(int K) { return (size_t)K * 4; }
__host__ __device__ inline size_t planes_code_bytes(int K) { return (size_t)K / 32; }

// Plane-0 scale code for a block with maximum magnitude amax.
__device__ __forceinline__ int planes_code0(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  const int ex = (int)(bits >> 23);
  if (ex == 0) return 1;   // zero or subnormal: the smallest normal scale covers it
  // amax = 2^(ex-127) * (1 + man/2^23); 6 * 2^(ex-129) = 1.5 * 2^(ex-127)
  const int c = (bits & 0x7FFFFFu) <= 0x400000u ? ex - 2 : ex - 1;
  return c < 1 ? 1 : c;
}

// E2M1 magnitude of code 0..7.
__device__ __forceinline__ float e2m1_value(uint32_t mag) {
  return mag < 4 ? 0.5f * (float)mag : (mag == 7 ? 6.0f : (float)mag - 2.0f);
}

// One warp, one 32-element block: lane i holds element i.  Writes the block's
// 128 plane bytes at `blk` with plane-0 code c0 (which must cover the block:
// 6 * 2^(c0-127) >= max |v|).
__device__ __forceinline__ void planes_block_c(float v, int lane, uint8_t* blk, int c0) {
  float r = v;
#pragma unroll
  for (int p = 0; p < kPlanes; ++p) {
    const int cp = max(c0 - 2 * p, 1);
    const float sp = __uint_as_float((uint32_t)cp << 23);
    const float t = r * __uint_as_float((uint32_t)(254 - cp) << 23);   // r / s_p, exact
    const uint32_t mag = e2m1_magnitude_code(fabsf(t));
    const bool neg = t < 0.0f;
    const uint32_t nib = mag | (neg && mag ? 8u : 0u);
    const float qv = e2m1_value(mag) * sp;
    r = neg ? r + qv : r - qv;
    // bytes: even lane L takes L and L + 1; words from lanes 8w, +2, +4, +6
    const uint32_t byte = nib | (__shfl_down_sync(0xffffffffu, nib, 1) << 4);
    const uint32_t b1 = __shfl_down_sync(0xffffffffu, byte, 2);
    const uint32_t b2 = __shfl_down_sync(0xffffffffu, byte, 4);
    const uint32_t b3 = __shfl_down_sync(0xffffffffu, byte, 6);
    if ((lane & 7) == 0)
      *reinterpret_cast<uint32_t*>(blk + p * 16 + lane / 2) =
          (byte & 0xFFu) | (b1 & 0xFFu) << 8 | (b2 & 0xFFu) << 16 | (b3 & 0xFFu) << 24;
  }
}

// The same with the block's own code (from its max |v|), which it returns.
__device__ __forceinline__ int planes_block(float v, int lane, uint8_t* blk) {
  const int c0 = planes_code0(warp_max(fabsf(v)));
  planes_block_c(v, lane, blk, c0);
  return c0;
}

// Bits of max |v| over a bf16 row of K elements (K / 8 a multiple of 32),
// this warp's share: lane entry i0, i0 + stride, ... of the row's K / 8 chunks
// of 8 elements, reduced over the warp (stride a multiple of 32, so every lane
// runs the same iterations).  f8: of the row's MXFP8 rounding instead (a lane
// quad holds one 32-element block).  The bits of a non-negative float.
__device__ __forceinline__ uint32_t row_amax_bits(const uint16_t* row, int K, int i0, int stride,
                                                  int f8) {
  const uint4* xr = reinterpret_cast<const uint4*>(row);
  uint32_t mx = 0;
  for (int i = i0; i < K / 8; i += stride) {
    const uint4 v = xr[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (f8) {
      float4 f0 = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                              __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
      float4 f1 = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                              __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
      mxfp8_round8(f0, f1);
      const float m = fmaxf(fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f0.z), fabsf(f0.w))),
                            fmaxf(fmaxf(fabsf(f1.x), fabsf(f1.y)), fmaxf(fabsf(f1.z), fabsf(f1.w))));
      mx = max(mx, __float_as_uint(m));
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
    }
  }
  if (!f8) mx <<= 16;   // bf16 magnitude bits -> float bits
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  return mx;
}

// Scale code of plane p given the block's plane-0 code.
__device__ __forceinline__ uint32_t planes_code(uint32_t c0, int p) {
  const int c = (int)c0 - 2 * p;
  return (uint32_t)(c < 1 ? 1 : c);
}

}  // namespace moe
