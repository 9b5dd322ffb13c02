// MXFP4 packing (host and device) and the debug dequantiser.
//
// Encoding (OCP Microscaling Formats (MX) v1.0): E2M1 elements, one E8M0 scale
// per 32 contiguous K elements.  Scale exponent = floor(log2 amax) - 2,
// clamped to [-127, 127] (an all-zero block takes -127), so amax / 2^e lies in
// [4, 8).  Each element w / 2^e (exact: a power-of-two scaling) is rounded to
// the E2M1 grid {0, .5, 1, 1.5, 2, 3, 4, 6} to nearest, ties to the even code,
// saturating at 6; the sign bit is the sign of w.  Canonical layout: byte j of
// a row holds elements 2j (low nibble) and 2j + 1 (high nibble).
//
// Kernel (tiled) layouts keep the same bytes, rearranged for the tensor-core
// consumers: rows go in tiles of 16 mma rows (layout 1: 16 consecutive rows;
// layout 2, for a [2n][k] gate/up matrix: gate rows 8T..8T+7 as mma rows 0..7
// and the matching up rows n+8T.. as mma rows 8..15).  Within a tile, the 16
// bytes lane L = 4g + t loads for K blocks 2P and 2P+1 are adjacent: bytes
// [4t, 4t+4) of mma rows g and g+8 in block 2P, then the same in block 2P+1.
// The scales of a tile are grouped by 4 blocks: for group Q and g < 8, eight
// bytes hold (row g, row g+8) for blocks 4Q..4Q+3.
//
// UMMA layouts (the tcgen05 block-scaled operand in shared memory, no swizzle,
// K-major): tiles of 128 mma rows (layout 3: 128 consecutive rows; layout 4,
// for a [2n][k] gate/up matrix: gate rows 64T..64T+63 as mma rows 0..63 and
// the matching up rows n+64T.. as mma rows 64..127).  A tile's nibbles are
// 8-row x 16-byte core matrices: the 16 bytes of K block b of mma row m sit at
// b*2048 + (m/8)*128 + (m%8)*16 (so one K block of the tile is 2 KB and any
// run of K blocks is contiguous).  A tile's scales come in atoms of 4 K
// blocks, 512 bytes each, in the order the 32x128b tensor-memory copy takes
// them: the scale of (m, b) at (b/4)*512 + (m%32)*16 + (m/32)*4 + b%4.
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

enum { kMxCanonical = 0, kMxTiled = 1, kMxTiledPairs = 2, kMxUmma = 3, kMxUmmaPairs = 4 };

__host__ __device__ inline bool mx_is_umma(int layout) {
  return layout == kMxUmma || layout == kMxUmmaPairs;
}

// Tile T and mma row r of canonical row `row` in a tiled or UMMA layout.
__host__ __device__ inline void mx_tile_of_row(int64_t row, int64_t rows, int layout, int64_t& T,
                                               int& r) {
  if (layout == kMxUmmaPairs) {
    const int64_t n = rows / 2;
    const int64_t i = row < n ? row : row - n;
    T = i / 64;
    r = (int)(i % 64) + (row < n ? 0 : 64);
  } else if (layout == kMxUmma) {
    T = row / 128;
    r = (int)(row % 128);
  } else if (layout == kMxTiledPairs) {
    const int64_t n = rows / 2;
    const int64_t i = row < n ? row : row - n;
    T = i / 8;
    r = (int)(i % 8) + (row < n ? 0 : 8);
  } else {
    T = row / 16;
    r = (int)(row % 16);
  }
}

// Byte offset of nibble bytes [4u, 4u+4) of K block b of (tile T, mma row r).
__host__ __device__ inline int64_t mx_tiled_word_offset(int64_t T, int r, int64_t b, int u,
                                                        int64_t k) {
  const int g = r & 7, half = r >> 3;
  return T * 8 * k + ((b / 2) * 32 + 4 * g + u) * 16 + (b % 2) * 8 + half * 4;
}

// Byte offset of the scale of K block b of (tile T, mma row r).
__host__ __device__ inline int64_t mx_tiled_scale_offset(int64_t T, int r, int64_t b, int64_t k) {
  const int g = r & 7, half = r >> 3;
  return T * (k / 2) + ((b / 4) * 8 + g) * 8 + (b % 4) * 2 + half;
}

// UMMA layouts: byte offset of the 16 nibble bytes / of the scale of K block
// b of (tile T, mma row m).
__host__ __device__ inline int64_t mx_umma_block_offset(int64_t T, int m, int64_t b, int64_t k) {
  return T * 64 * k + b * 2048 + (m / 8) * 128 + (m % 8) * 16;
}
__host__ __device__ inline int64_t mx_umma_scale_offset(int64_t T, int m, int64_t b, int64_t k) {
  return T * 4 * k + (b / 4) * 512 + (m % 32) * 16 + (m / 32) * 4 + b % 4;
}

// Where the 16 nibble bytes and the scale byte of (row, block b) go.
__host__ __device__ inline void mx_store_block(uint8_t* q, uint8_t* s, int64_t row, int64_t b,
                                               int64_t rows, int64_t k, int layout,
                                               const uint8_t (&qb)[16], uint8_t sb) {
  if (layout == kMxCanonical) {
    memcpy(q + row * (k / 2) + b * 16, qb, 16);
    s[row * (k / 32) + b] = sb;
    return;
  }
  if (mx_is_umma(layout)) {
    int64_t T;
    int m;
    mx_tile_of_row(row, rows, layout, T, m);
    memcpy(q + mx_umma_block_offset(T, m, b, k), qb, 16);
    s[mx_umma_scale_offset(T, m, b, k)] = sb;
    return;
  }
  int64_t T;
  int r;
  mx_tile_of_row(row, rows, layout, T, r);
  for (int u = 0; u < 4; ++u) memcpy(q + mx_tiled_word_offset(T, r, b, u, k), qb + 4 * u, 4);
  s[mx_tiled_scale_offset(T, r, b, k)] = sb;
}

// The 16 nibble bytes and the scale byte of (row, block b) in a layout.
__host__ __device__ inline uint8_t mx_load_block(const uint8_t* q, const uint8_t* s, int64_t row,
                                                 int64_t b, int64_t rows, int64_t k, int layout,
                                                 uint8_t (&qb)[16]) {
  if (layout == kMxCanonical) {
    memcpy(qb, q + row * (k / 2) + b * 16, 16);
    return s[row * (k / 32) + b];
  }
  if (mx_is_umma(layout)) {
    int64_t T;
    int m;
    mx_tile_of_row(row, rows, layout, T, m);
    memcpy(qb, q + mx_umma_block_offset(T, m, b, k), 16);
    return s[mx_umma_scale_offset(T, m, b, k)];
  }
  int64_t T;
  int r;
  mx_tile_of_row(row, rows, layout, T, r);
  for (int u = 0; u < 4; ++u) memcpy(qb + 4 * u, q + mx_tiled_word_offset(T, r, b, u, k), 4);
  return s[mx_tiled_scale_offset(T, r, b, k)];
}

// A layout's shape rules: k % 32 (canonical); tiled and UMMA layouts also
// k % 128 and whole tiles (16 rows tiled, 128 rows UMMA).
__host__ __device__ inline bool mx_layout_ok(int64_t rows, int64_t k, int layout) {
  if (rows < 0 || k <= 0 || k % 32 != 0) return false;
  if (layout == kMxCanonical) return true;
  if (mx_is_umma(layout)) return k % 128 == 0 && rows % 128 == 0;
  if (layout != kMxTiled && layout != kMxTiledPairs) return false;
  return k % 128 == 0 && rows % 16 == 0;
}

__global__ void mxfp4_pack_kernel(const float* __restrict__ w, int64_t rows, int64_t k,
                                  uint8_t* __restrict__ q, uint8_t* __restrict__ s, int layout) {
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
    const uint8_t sb = mx_pack_block(blk, qb);
    mx_store_block(q, s, r, b, rows, k, layout, qb, sb);
  }
}

// Canonical packed bytes -> a tiled layout (a byte permutation).
__global__ void mxfp4_retile_kernel(const uint8_t* __restrict__ qc, const uint8_t* __restrict__ sc,
                                    int64_t rows, int64_t k, uint8_t* __restrict__ q,
                                    uint8_t* __restrict__ s, int layout) {
  const int64_t nb = k / 32;
  const int64_t total = rows * nb;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / nb, b = t % nb;
    uint8_t qb[16];
    const uint4 v = *reinterpret_cast<const uint4*>(qc + r * (k / 2) + b * 16);
    memcpy(qb, &v, 16);
    mx_store_block(q, s, r, b, rows, k, layout, qb, sc[r * nb + b]);
  }
}

// Any layout -> any layout (a byte permutation).
__global__ void mxfp4_relayout_kernel(const uint8_t* __restrict__ qi, const uint8_t* __restrict__ si,
                                      int64_t rows, int64_t k, int from, uint8_t* __restrict__ q,
                                      uint8_t* __restrict__ s, int to) {
  const int64_t nb = k / 32;
  const int64_t total = rows * nb;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / nb, b = t % nb;
    uint8_t qb[16];
    const uint8_t sb = mx_load_block(qi, si, r, b, rows, k, from, qb);
    mx_store_block(q, s, r, b, rows, k, to, qb, sb);
  }
}

// Dequantise rows x k (any layout) into canonical fp32 rows with the
// consumers' element decode (cvt.rn.f16x2.e2m1x2) and the exact E8M0 value.
__global__ void mxfp4_dequant_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                     int64_t rows, int64_t k, int layout,
                                     float* __restrict__ out) {
  const int64_t nb = k / 32;
  const int64_t total = rows * nb;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / nb, b = t % nb;
    uint32_t words[4];
    float sc;
    if (layout == kMxCanonical) {
      const uint4 v = *reinterpret_cast<const uint4*>(q + r * (k / 2) + b * 16);
      words[0] = v.x;
      words[1] = v.y;
      words[2] = v.z;
      words[3] = v.w;
      sc = e8m0_to_f32(s[r * nb + b]);
    } else if (mx_is_umma(layout)) {
      int64_t T;
      int mr;
      mx_tile_of_row(r, rows, layout, T, mr);
      const uint4 v = *reinterpret_cast<const uint4*>(q + mx_umma_block_offset(T, mr, b, k));
      words[0] = v.x;
      words[1] = v.y;
      words[2] = v.z;
      words[3] = v.w;
      sc = e8m0_to_f32(s[mx_umma_scale_offset(T, mr, b, k)]);
    } else {
      int64_t T;
      int mr;
      mx_tile_of_row(r, rows, layout, T, mr);
      for (int u = 0; u < 4; ++u)
        words[u] = *reinterpret_cast<const uint32_t*>(q + mx_tiled_word_offset(T, mr, b, u, k));
      sc = e8m0_to_f32(s[mx_tiled_scale_offset(T, mr, b, k)]);
    }
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
