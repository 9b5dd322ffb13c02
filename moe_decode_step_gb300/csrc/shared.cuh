// Shared expert: bf16 SwiGLU GEMV on a side stream, overlapping the router and
// the routed experts ("Kimi K3 on GB300: 13 kernels a layer...", section "What
// the fused path changes": the shared expert runs on a side stream).
//
// Same K-split shape as the routed kernels: KW warps split K, each lane keeps
// its activation slice in registers and streams 16-byte weight loads.
//  FC1: lane owns 32 elements (4 loads per row); x stays bf16 and products use
//       the mixed fma.rn.f32.bf16 (exact products, fp32 sums).
//  FC2: lane owns 16 elements (2 loads per row); the fp32 h_s slice stays in
//       registers and bf16 weights widen exactly to fp32 for FFMA.
#pragma once

#include "common.cuh"

namespace moe {

struct SharedArgs {
  const uint16_t* w;     // FC1: bf16 [2F][d]; FC2: bf16 [d][F]
  int K;                 // row length
  int N;                 // outputs (FC1: F row pairs, FC2: d rows)
  int B;                 // rows of activations
  const uint16_t* x;     // FC1 activations bf16 [B][d]
  const float* hs;       // FC2 activations fp32 [B][F]
  float* out;            // FC1: hs [B][F]; FC2: y_s [B][d]
};

constexpr int kSh1UB = 2;   // row pairs per batch (16 loads in flight per lane)
constexpr int kSh1NB = 2;
constexpr int kSh1RPW = kSh1UB * kSh1NB;

template <int R>
__device__ __forceinline__ void sh1_pass(const SharedArgs& a, int b0, int i_item, int kw, int KW,
                                         int rg, int RG, int lane, float* s_red) {
  const int c = kw * 32 + lane;              // 32-element chunk index
  const bool lane_ok = c < a.K / 32;
  uint32_t xa[R][16];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint4* p = reinterpret_cast<const uint4*>(a.x + (size_t)(b0 + r) * a.K + c * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = lane_ok ? p[q] : make_uint4(0, 0, 0, 0);
      xa[r][q * 4 + 0] = v.x;
      xa[r][q * 4 + 1] = v.y;
      xa[r][q * 4 + 2] = v.z;
      xa[r][q * 4 + 3] = v.w;
    }
  }
  const int i_grp = i_item + rg * kSh1RPW;
  constexpr int V = kSh1UB * R * 2;
  constexpr int M = (V == 4) ? 2 : (V == 8) ? 3 : 4;
#pragma unroll
  for (int nb = 0; nb < kSh1NB; ++nb) {
    uint4 wg[kSh1UB][4], wu[kSh1UB][4];
#pragma unroll
    for (int u = 0; u < kSh1UB; ++u) {
      const int i = i_grp + nb * kSh1UB + u;
      const bool ok = lane_ok && i < a.N;
      const uint16_t* rg_ = a.w + (size_t)i * a.K + c * 32;
      const uint16_t* ru_ = a.w + (size_t)(a.N + i) * a.K + c * 32;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        wg[u][q] = ok ? ld_stream_u128(rg_ + q * 8) : make_uint4(0, 0, 0, 0);
        wu[u][q] = ok ? ld_stream_u128(ru_ + q * 8) : make_uint4(0, 0, 0, 0);
      }
    }
    float v[V];
#pragma unroll
    for (int u = 0; u < kSh1UB; ++u) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float sg = 0.f, su = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          sg = fma2_bf16(wg[u][q].x, xa[r][q * 4 + 0], sg);
          sg = fma2_bf16(wg[u][q].y, xa[r][q * 4 + 1], sg);
          sg = fma2_bf16(wg[u][q].z, xa[r][q * 4 + 2], sg);
          sg = fma2_bf16(wg[u][q].w, xa[r][q * 4 + 3], sg);
          su = fma2_bf16(wu[u][q].x, xa[r][q * 4 + 0], su);
          su = fma2_bf16(wu[u][q].y, xa[r][q * 4 + 1], su);
          su = fma2_bf16(wu[u][q].z, xa[r][q * 4 + 2], su);
          su = fma2_bf16(wu[u][q].w, xa[r][q * 4 + 3], su);
        }
        v[(u * R + r) * 2 + 0] = sg;
        v[(u * R + r) * 2 + 1] = su;
      }
    }
    const float sum = warp_reduce_scatter<V>(v, lane);
    if ((lane & ((1 << (5 - M)) - 1)) == 0) {
      const int vi = lane >> (5 - M);
      const int u = vi / (R * 2), r = (vi / 2) % R, gu = vi & 1;
      const int rp = nb * kSh1UB + u;
      s_red[(((rg * kSh1RPW + rp) * 4 + r) * 2 + gu) * KW + kw] = sum;
    }
  }
  __syncthreads();
  const int n_out = RG * kSh1RPW * R;
  for (int t = threadIdx.x; t < n_out; t += blockDim.x) {
    const int r = t % R, rp = (t / R) % kSh1RPW, g = t / (R * kSh1RPW);
    const int i = i_item + g * kSh1RPW + rp;
    if (i < a.N) {
      const float* pg = s_red + (((g * kSh1RPW + rp) * 4 + r) * 2 + 0) * KW;
      const float* pu = pg + KW;
      float sg = 0.f, su = 0.f;
      for (int w = 0; w < KW; ++w) { sg += pg[w]; su += pu[w]; }
      a.out[(size_t)(b0 + r) * a.N + i] = sg / (1.0f + expf(-sg)) * su;
    }
  }
  __syncthreads();
}

template <int RMAX>
__global__ void __launch_bounds__(256)
shared_fc1_kernel(const SharedArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = (a.K + 1023) / 1024;
  const int RG = blockDim.x / 32 / KW;
  const int kw = warp % KW, rg = warp / KW;
  __shared__ float s_red[8 * kSh1RPW * 4 * 2];
  const int rows_per_item = RG * kSh1RPW;
  const int n_items = (a.N + rows_per_item - 1) / rows_per_item;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int i_item = it * rows_per_item;
    for (int b0 = 0; b0 < a.B;) {
      const int left = a.B - b0;
      if (RMAX >= 4 && left >= 4) {
        if constexpr (RMAX >= 4) sh1_pass<4>(a, b0, i_item, kw, KW, rg, RG, lane, s_red);
        b0 += 4;
      } else if (RMAX >= 2 && left >= 2) {
        if constexpr (RMAX >= 2) sh1_pass<2>(a, b0, i_item, kw, KW, rg, RG, lane, s_red);
        b0 += 2;
      } else {
        sh1_pass<1>(a, b0, i_item, kw, KW, rg, RG, lane, s_red);
        b0 += 1;
      }
    }
  }
}

constexpr int kSh2UB = 8;    // rows per batch (16 loads in flight per lane)
constexpr int kSh2NB = 2;
constexpr int kSh2RPW = kSh2UB * kSh2NB;

template <int R>
__device__ __forceinline__ void sh2_pass(const SharedArgs& a, int b0, int n_item, int kw, int KW,
                                         int rg, int RG, int lane, float* s_red) {
  const int c = kw * 32 + lane;              // 16-element chunk index
  const bool lane_ok = c < a.K / 16;
  float ha[R][16];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float4* p = reinterpret_cast<const float4*>(a.hs + (size_t)(b0 + r) * a.K + c * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = lane_ok ? __ldcg(p + q) : make_float4(0.f, 0.f, 0.f, 0.f);
      ha[r][q * 4 + 0] = v.x;
      ha[r][q * 4 + 1] = v.y;
      ha[r][q * 4 + 2] = v.z;
      ha[r][q * 4 + 3] = v.w;
    }
  }
  const int n_grp = n_item + rg * kSh2RPW;
  constexpr int V = kSh2UB * R;
  constexpr int M = (V == 8) ? 3 : (V == 16) ? 4 : 5;
#pragma unroll
  for (int nb = 0; nb < kSh2NB; ++nb) {
    uint4 w[kSh2UB][2];
#pragma unroll
    for (int u = 0; u < kSh2UB; ++u) {
      const int n = n_grp + nb * kSh2UB + u;
      const bool ok = lane_ok && n < a.N;
      const uint16_t* row = a.w + (size_t)n * a.K + c * 16;
      w[u][0] = ok ? ld_stream_u128(row) : make_uint4(0, 0, 0, 0);
      w[u][1] = ok ? ld_stream_u128(row + 8) : make_uint4(0, 0, 0, 0);
    }
    float v[V];
#pragma unroll
    for (int u = 0; u < kSh2UB; ++u) {
      const uint32_t ww[8] = {w[u][0].x, w[u][0].y, w[u][0].z, w[u][0].w,
                              w[u][1].x, w[u][1].y, w[u][1].z, w[u][1].w};
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          s0 = fmaf(__uint_as_float(ww[t] << 16), ha[r][2 * t], s0);
          s1 = fmaf(__uint_as_float(ww[t] & 0xFFFF0000u), ha[r][2 * t + 1], s1);
        }
        v[u * R + r] = s0 + s1;
      }
    }
    const float sum = warp_reduce_scatter<V>(v, lane);
    if ((lane & ((1 << (5 - M)) - 1)) == 0) {
      const int vi = lane >> (5 - M);
      const int u = vi / R, r = vi % R;
      const int rr = nb * kSh2UB + u;
      s_red[((rg * kSh2RPW + rr) * 4 + r) * KW + kw] = sum;
    }
  }
  __syncthreads();
  const int n_out = RG * kSh2RPW * R;
  for (int t = threadIdx.x; t < n_out; t += blockDim.x) {
    const int r = t % R, rr = (t / R) % kSh2RPW, g = t / (R * kSh2RPW);
    const int n = n_item + g * kSh2RPW + rr;
    if (n < a.N) {
      const float* pp = s_red + ((g * kSh2RPW + rr) * 4 + r) * KW;
      float acc = 0.f;
      for (int w2 = 0; w2 < KW; ++w2) acc += pp[w2];
      a.out[(size_t)(b0 + r) * a.N + n] = acc;
    }
  }
  __syncthreads();
}

template <int RMAX>
__global__ void __launch_bounds__(256)
shared_fc2_kernel(const SharedArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = (a.K + 511) / 512;
  const int RG = blockDim.x / 32 / KW;
  const int kw = warp % KW, rg = warp / KW;
  __shared__ float s_red[8 * kSh2RPW * 4];
  const int rows_per_item = RG * kSh2RPW;
  const int n_items = (a.N + rows_per_item - 1) / rows_per_item;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int n_item = it * rows_per_item;
    for (int b0 = 0; b0 < a.B;) {
      const int left = a.B - b0;
      if (RMAX >= 4 && left >= 4) {
        if constexpr (RMAX >= 4) sh2_pass<4>(a, b0, n_item, kw, KW, rg, RG, lane, s_red);
        b0 += 4;
      } else if (RMAX >= 2 && left >= 2) {
        if constexpr (RMAX >= 2) sh2_pass<2>(a, b0, n_item, kw, KW, rg, RG, lane, s_red);
        b0 += 2;
      } else {
        sh2_pass<1>(a, b0, n_item, kw, KW, rg, RG, lane, s_red);
        b0 += 1;
      }
    }
  }
}

}  // namespace moe
