// Routed experts: MXFP4 dequant-GEMV, FC1 (gate/up + SwiGLU) and FC2 (down).
//
// Role from "Kimi K3 on GB300: 13 kernels a layer...", section "What the fused
// path changes": the routed experts run as persistent kernels doing FC1 and
// FC2 over all selected experts; packed FP4 weights are streamed from HBM
// ("Why batch 1 on a rack is not only a bandwidth problem": about one FLOP per
// byte, so the path is bound by HBM, not by the tensor cores).
//
// Design (one GB300, B = 1..64 rows):
//  * Work item = (active expert, tile of output rows).  CTAs pull items from a
//    device counter, so CTAs that start late (the shared expert occupies SMs
//    at first) simply take fewer items.
//  * Inside a CTA, KW warps split K: lane l of warp w owns K elements
//    [(w*32 + l) * EPL, +EPL): one MX block (FC1, 16-byte loads) or half a block
//    (FC2, 8-byte loads).  The activation slice of a lane stays in registers as
//    f16x2 for the whole item, so weights are the only streamed operand.
//  * E2M1 -> f16x2 by cvt.rn.f16x2.e2m1x2 (exact), products by the mixed
//    fma.rn.f32.f16 (exact products, fp32 sums), the E8M0 scale applied once
//    per block.  Activations are scaled by 2^-shift (shift = 0 unless
//    |a| >= 2^15) so they never overflow f16; results are scaled back exactly.
//  * Per-lane block partials are combined with a butterfly reduce-scatter and
//    then across the KW warps in shared memory, in a fixed order (no float
//    atomics: results are deterministic).
#pragma once

#include "common.cuh"

namespace moe {

struct RoutedArgs {
  const uint8_t* q;          // nibbles of expert 0; expert e at q + e * q_stride
  const uint8_t* s;          // scale bytes of expert 0
  size_t q_stride, s_stride; // bytes per expert
  int K;                     // row length (FC1: d, FC2: f)
  int N;                     // outputs per expert (FC1: f row pairs, FC2: d rows)
  int k;                     // top-k (pair p belongs to row p / k)
  const uint16_t* x;         // FC1 activations: bf16 [B][d]
  const int* x_shift;        // [B]
  const float* h;            // FC2 activations: fp32 [P][f]
  const unsigned* h_amax;    // [P] bits of max |h|
  float* out;                // FC1: h [P][f]; FC2: y_pair [P][d]
  unsigned* out_amax;        // FC1: h_amax [P]
  const int* n_active;
  const int* active_expert;
  const int* active_off;
  const int* pair_list;
  int* work;                 // item counter (0 at launch)
};

// Pull the next item for the whole CTA; returns -1 when done.
__device__ __forceinline__ int next_item(int* counter, int n_items, int* s_slot) {
  __syncthreads();
  if (threadIdx.x == 0) *s_slot = atomicAdd(counter, 1);
  __syncthreads();
  const int it = *s_slot;
  return it < n_items ? it : -1;
}

// ---------------------------------------------------------------------------
// FC1: h[p][i] = silu(W_g[i] . x_b) * (W_u[i] . x_b) for the pairs p of expert e.
// ---------------------------------------------------------------------------
constexpr int kFc1UB = 4;    // row pairs per load batch
constexpr int kFc1NB = 4;    // batches per item (per row group)
constexpr int kFc1RPW = kFc1UB * kFc1NB;

struct Fc1Batch {
  uint4 g[kFc1UB], u[kFc1UB];
  uint32_t sg[kFc1UB], su[kFc1UB];
};

__device__ __forceinline__ void fc1_load(const uint8_t* qe, const uint8_t* se, int K, int N, int i0,
                                         int blk, bool lane_ok, Fc1Batch& bt) {
#pragma unroll
  for (int u = 0; u < kFc1UB; ++u) {
    const int i = i0 + u;
    if (lane_ok && i < N) {
      bt.g[u] = ld_stream_u128(qe + (size_t)i * (K / 2) + blk * 16);
      bt.u[u] = ld_stream_u128(qe + (size_t)(N + i) * (K / 2) + blk * 16);
      bt.sg[u] = ld_stream_u8(se + (size_t)i * (K / 32) + blk);
      bt.su[u] = ld_stream_u8(se + (size_t)(N + i) * (K / 32) + blk);
    } else {
      bt.g[u] = bt.u[u] = make_uint4(0, 0, 0, 0);
      bt.sg[u] = bt.su[u] = 0;
    }
  }
}

// Dot of one 32-element MX block (16 bytes) with R activation slices.
template <int R>
__device__ __forceinline__ void mx_block_dot(const uint4& wq, const uint32_t (&xa)[R][16],
                                             float (&part)[R]) {
#pragma unroll
  for (int r = 0; r < R; ++r) part[r] = 0.f;
  const uint32_t words[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t hq[4];
    e2m1x8_to_f16x2(words[w], hq);
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int t = 0; t < 4; ++t) part[r] = fma2_f16(hq[t], xa[r][w * 4 + t], part[r]);
    }
  }
}

template <int R>
__device__ __forceinline__ void fc1_compute(const Fc1Batch& bt, const uint32_t (&xa)[R][16],
                                            float (&v)[kFc1UB * R * 2]) {
#pragma unroll
  for (int u = 0; u < kFc1UB; ++u) {
    float pg[R], pu[R];
    mx_block_dot<R>(bt.g[u], xa, pg);
    mx_block_dot<R>(bt.u[u], xa, pu);
    const float scg = e8m0_to_f32(bt.sg[u]), scu = e8m0_to_f32(bt.su[u]);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      v[(u * R + r) * 2 + 0] = pg[r] * scg;
      v[(u * R + r) * 2 + 1] = pu[r] * scu;
    }
  }
}

// Load the lane's 32-element x slice of row b as f16x2, scaled by 2^-shift.
__device__ __forceinline__ void load_x_f16(const uint16_t* xrow, int blk, bool lane_ok, int shift,
                                           uint32_t (&xa)[16]) {
  if (!lane_ok) {
#pragma unroll
    for (int t = 0; t < 16; ++t) xa[t] = 0;
    return;
  }
  const float sc = pow2f(-shift);
  const uint4* p = reinterpret_cast<const uint4*>(xrow + blk * 32);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = p[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float lo = __uint_as_float(w[t] << 16) * sc;
      const float hi = __uint_as_float(w[t] & 0xFFFF0000u) * sc;
      xa[c * 4 + t] = pack_f16x2(lo, hi);
    }
  }
}

// One pass over R (1, 2 or 4) pairs of expert e for the item's row pairs.
// s_red layout: [rg][row pair in group][r][gate/up][kw]
template <int R>
__device__ __forceinline__ void fc1_pass(const RoutedArgs& a, const uint8_t* qe, const uint8_t* se,
                                         const int* s_pairs, int i_item, int kw, int KW, int rg,
                                         int RG, int lane, float* s_red, unsigned* s_amax) {
  const int blk = kw * 32 + lane;
  const bool lane_ok = blk < a.K / 32;
  uint32_t xa[R][16];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int b = s_pairs[r] / a.k;
    load_x_f16(a.x + (size_t)b * a.K, blk, lane_ok, a.x_shift[b], xa[r]);
  }
  const int i_grp = i_item + rg * kFc1RPW;
  constexpr int V = kFc1UB * R * 2;
  constexpr int M = (V == 8) ? 3 : (V == 16) ? 4 : 5;
  Fc1Batch cur, nxt;
  fc1_load(qe, se, a.K, a.N, i_grp, blk, lane_ok, cur);
#pragma unroll
  for (int nb = 0; nb < kFc1NB; ++nb) {
    if (nb + 1 < kFc1NB) fc1_load(qe, se, a.K, a.N, i_grp + (nb + 1) * kFc1UB, blk, lane_ok, nxt);
    float v[V];
    fc1_compute<R>(cur, xa, v);
    const float sum = warp_reduce_scatter<V>(v, lane);
    if ((lane & ((1 << (5 - M)) - 1)) == 0) {
      const int vi = lane >> (5 - M);          // (u * R + r) * 2 + gu
      const int u = vi / (R * 2), r = (vi / 2) % R, gu = vi & 1;
      const int rp = nb * kFc1UB + u;
      s_red[(((rg * kFc1RPW + rp) * 4 + r) * 2 + gu) * KW + kw] = sum;
    }
    if (nb + 1 < kFc1NB) cur = nxt;
  }
  __syncthreads();
  // finalize: one thread per (rg, row pair, r)
  const int n_out = RG * kFc1RPW * R;
  for (int t = threadIdx.x; t < n_out; t += blockDim.x) {
    const int r = t % R, rp = (t / R) % kFc1RPW, g = t / (R * kFc1RPW);
    const int i = i_item + g * kFc1RPW + rp;
    if (i < a.N) {
      float sg = 0.f, su = 0.f;
      const float* pg = s_red + (((g * kFc1RPW + rp) * 4 + r) * 2 + 0) * KW;
      const float* pu = pg + KW;
      for (int w = 0; w < KW; ++w) { sg += pg[w]; su += pu[w]; }
      const int p = s_pairs[r];
      const float back = pow2f(a.x_shift[p / a.k]);
      const float gg = sg * back, uu = su * back;
      const float hv = gg / (1.0f + expf(-gg)) * uu;
      a.out[(size_t)p * a.N + i] = hv;
      atomicMax(&s_amax[r], __float_as_uint(fabsf(hv)));
    }
  }
  __syncthreads();
  if (threadIdx.x < R) {
    atomicMax(&a.out_amax[s_pairs[threadIdx.x]], s_amax[threadIdx.x]);
    s_amax[threadIdx.x] = 0u;
  }
}

template <int RMAX>
__global__ void __launch_bounds__(256)
routed_fc1_kernel(const RoutedArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = (a.K + 1023) / 1024;
  const int RG = blockDim.x / 32 / KW;
  const int kw = warp % KW, rg = warp / KW;
  __shared__ float s_red[8 * kFc1RPW * 4 * 2];   // >= RG*RPW*4*2*KW for RG*KW <= 8
  __shared__ int s_pairs[4];
  __shared__ unsigned s_amax[4];
  __shared__ int s_slot;
  if (threadIdx.x < 4) s_amax[threadIdx.x] = 0u;
  const int n_act = *a.n_active;
  const int rows_per_item = RG * kFc1RPW;
  const int tiles = (a.N + rows_per_item - 1) / rows_per_item;
  const int n_items = n_act * tiles;
  for (int it = next_item(a.work, n_items, &s_slot); it >= 0;
       it = next_item(a.work, n_items, &s_slot)) {
    const int slot = it / tiles, tile = it % tiles;
    const int e = a.active_expert[slot];
    const int p0 = a.active_off[slot], pr = a.active_off[slot + 1] - p0;
    const uint8_t* qe = a.q + (size_t)e * a.q_stride;
    const uint8_t* se = a.s + (size_t)e * a.s_stride;
    const int i_item = tile * rows_per_item;
    for (int done = 0; done < pr;) {
      int R = pr - done;
      R = R >= 4 ? 4 : (R >= 2 ? 2 : 1);
      if (R > RMAX) R = RMAX;
      __syncthreads();
      if (threadIdx.x < R) s_pairs[threadIdx.x] = a.pair_list[p0 + done + threadIdx.x];
      __syncthreads();
      if (R == 1) fc1_pass<1>(a, qe, se, s_pairs, i_item, kw, KW, rg, RG, lane, s_red, s_amax);
      if constexpr (RMAX >= 2) {
        if (R == 2) fc1_pass<2>(a, qe, se, s_pairs, i_item, kw, KW, rg, RG, lane, s_red, s_amax);
      }
      if constexpr (RMAX >= 4) {
        if (R == 4) fc1_pass<4>(a, qe, se, s_pairs, i_item, kw, KW, rg, RG, lane, s_red, s_amax);
      }
      done += R;
    }
  }
}

// ---------------------------------------------------------------------------
// FC2: y_pair[p][n] = W_d[n] . h_p for the pairs p of expert e.
// Lane owns 16 elements (half an MX block, 8-byte loads).
// ---------------------------------------------------------------------------
constexpr int kFc2UB = 16;   // rows per load batch
constexpr int kFc2NB = 2;    // batches per item (per row group)
constexpr int kFc2RPW = kFc2UB * kFc2NB;

struct Fc2Batch {
  uint2 w[kFc2UB];
  uint32_t s[kFc2UB];
};

__device__ __forceinline__ void fc2_load(const uint8_t* qe, const uint8_t* se, int K, int N, int n0,
                                         int hb, bool lane_ok, Fc2Batch& bt) {
#pragma unroll
  for (int u = 0; u < kFc2UB; ++u) {
    const int n = n0 + u;
    if (lane_ok && n < N) {
      bt.w[u] = ld_stream_u64(qe + (size_t)n * (K / 2) + hb * 8);
      bt.s[u] = ld_stream_u8(se + (size_t)n * (K / 32) + (hb >> 1));
    } else {
      bt.w[u] = make_uint2(0, 0);
      bt.s[u] = 0;
    }
  }
}

template <int R>
__device__ __forceinline__ void fc2_compute(const Fc2Batch& bt, const uint32_t (&ha)[R][8],
                                            float (&v)[kFc2UB * R]) {
#pragma unroll
  for (int u = 0; u < kFc2UB; ++u) {
    float part[R];
#pragma unroll
    for (int r = 0; r < R; ++r) part[r] = 0.f;
    const uint32_t words[2] = {bt.w[u].x, bt.w[u].y};
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      uint32_t hq[4];
      e2m1x8_to_f16x2(words[w], hq);
#pragma unroll
      for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int t = 0; t < 4; ++t) part[r] = fma2_f16(hq[t], ha[r][w * 4 + t], part[r]);
      }
    }
    const float sc = e8m0_to_f32(bt.s[u]);
#pragma unroll
    for (int r = 0; r < R; ++r) v[u * R + r] = part[r] * sc;
  }
}

// Load the lane's 16-element slice of h_p as f16x2, scaled by 2^-shift.
__device__ __forceinline__ void load_h_f16(const float* hrow, int hb, bool lane_ok, int shift,
                                           uint32_t (&ha)[8]) {
  if (!lane_ok) {
#pragma unroll
    for (int t = 0; t < 8; ++t) ha[t] = 0;
    return;
  }
  const float sc = pow2f(-shift);
  const float4* p = reinterpret_cast<const float4*>(hrow + hb * 16);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float4 v = __ldcg(p + c);
    ha[c * 2 + 0] = pack_f16x2(v.x * sc, v.y * sc);
    ha[c * 2 + 1] = pack_f16x2(v.z * sc, v.w * sc);
  }
}

template <int R>
__device__ __forceinline__ void fc2_pass(const RoutedArgs& a, const uint8_t* qe, const uint8_t* se,
                                         const int* s_pairs, const int* s_shift, int n_item, int kw,
                                         int KW, int rg, int RG, int lane, float* s_red) {
  const int hb = kw * 32 + lane;
  const bool lane_ok = hb < a.K / 16;
  uint32_t ha[R][8];
#pragma unroll
  for (int r = 0; r < R; ++r)
    load_h_f16(a.h + (size_t)s_pairs[r] * a.K, hb, lane_ok, s_shift[r], ha[r]);
  const int n_grp = n_item + rg * kFc2RPW;
  constexpr int V = kFc2UB * R;
  constexpr int M = (V == 16) ? 4 : 5;
  Fc2Batch cur, nxt;
  fc2_load(qe, se, a.K, a.N, n_grp, hb, lane_ok, cur);
#pragma unroll
  for (int nb = 0; nb < kFc2NB; ++nb) {
    if (nb + 1 < kFc2NB) fc2_load(qe, se, a.K, a.N, n_grp + (nb + 1) * kFc2UB, hb, lane_ok, nxt);
    float v[V];
    fc2_compute<R>(cur, ha, v);
    const float sum = warp_reduce_scatter<V>(v, lane);
    if ((lane & ((1 << (5 - M)) - 1)) == 0) {
      const int vi = lane >> (5 - M);  // u * R + r
      const int u = vi / R, r = vi % R;
      const int rr = nb * kFc2UB + u;
      s_red[((rg * kFc2RPW + rr) * 2 + r) * KW + kw] = sum;
    }
    if (nb + 1 < kFc2NB) cur = nxt;
  }
  __syncthreads();
  const int n_out = RG * kFc2RPW * R;
  for (int t = threadIdx.x; t < n_out; t += blockDim.x) {
    const int r = t % R, rr = (t / R) % kFc2RPW, g = t / (R * kFc2RPW);
    const int n = n_item + g * kFc2RPW + rr;
    if (n < a.N) {
      const float* pp = s_red + ((g * kFc2RPW + rr) * 2 + r) * KW;
      float acc = 0.f;
      for (int w = 0; w < KW; ++w) acc += pp[w];
      a.out[(size_t)s_pairs[r] * a.N + n] = acc * pow2f(s_shift[r]);
    }
  }
}

template <int RMAX>
__global__ void __launch_bounds__(256)
routed_fc2_kernel(const RoutedArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = (a.K + 511) / 512;
  const int RG = blockDim.x / 32 / KW;
  const int kw = warp % KW, rg = warp / KW;
  __shared__ float s_red[8 * kFc2RPW * 2];   // >= RG*RPW*2*KW for RG*KW <= 8
  __shared__ int s_pairs[2], s_shift[2];
  __shared__ int s_slot;
  const int n_act = *a.n_active;
  const int rows_per_item = RG * kFc2RPW;
  const int tiles = (a.N + rows_per_item - 1) / rows_per_item;
  const int n_items = n_act * tiles;
  for (int it = next_item(a.work, n_items, &s_slot); it >= 0;
       it = next_item(a.work, n_items, &s_slot)) {
    const int slot = it / tiles, tile = it % tiles;
    const int e = a.active_expert[slot];
    const int p0 = a.active_off[slot], pr = a.active_off[slot + 1] - p0;
    const uint8_t* qe = a.q + (size_t)e * a.q_stride;
    const uint8_t* se = a.s + (size_t)e * a.s_stride;
    const int n_item = tile * rows_per_item;
    for (int done = 0; done < pr;) {
      int R = pr - done >= 2 ? 2 : 1;
      if (R > RMAX) R = RMAX;
      __syncthreads();
      if (threadIdx.x < R) {
        const int p = a.pair_list[p0 + done + threadIdx.x];
        s_pairs[threadIdx.x] = p;
        s_shift[threadIdx.x] = f16_shift_for_amax(__uint_as_float(__ldcg(a.h_amax + p)));
      }
      __syncthreads();
      if (R == 1) fc2_pass<1>(a, qe, se, s_pairs, s_shift, n_item, kw, KW, rg, RG, lane, s_red);
      if constexpr (RMAX >= 2) {
        if (R == 2) fc2_pass<2>(a, qe, se, s_pairs, s_shift, n_item, kw, KW, rg, RG, lane, s_red);
      }
      done += R;
    }
  }
}

}  // namespace moe
