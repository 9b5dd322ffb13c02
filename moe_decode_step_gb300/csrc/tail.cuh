// MoE tail: weighted combine of the routed experts + shared expert + residual,
// then RMSNorm, in one kernel ("Kimi K3 on GB300: 13 kernels a layer...",
// section "What the fused path changes": the tail folds the down-projection
// reduction and the next norm together; at one GPU the reduction is local).
//
// Grid (S, B): CTA (s, b) owns 256 elements of row b.  It forms
//   z = residual + sum_j w[b][j] * y_pair[b*k + j] + y_s,
// writes residual <- bf16(z) and the fp32 z, and a partial sum of squares.
// The last CTA of the row (atomic ticket, no waiting) adds the S partials in
// slice order and writes out = bf16(z / sqrt(mean z^2 + eps) * gamma).
#pragma once

#include "common.cuh"

namespace moe {

struct TailArgs {
  const float* y_pair;     // [B*k][d]
  const float* topk_w;     // [B][k]
  const float* y_s;        // [B][d]
  const uint16_t* gamma;   // bf16 [d]
  uint16_t* residual;      // bf16 [B][d] in / out
  uint16_t* out;           // bf16 [B][d]
  float* z;                // workspace [B][d]
  float* psum;             // workspace [B][S]
  unsigned* ticket;        // workspace [B], 0 at rest
  float* y_r_dbg;          // optional export [B][d]
  float* out_dbg;          // optional export of out before bf16 rounding [B][d]
  int B, d, k;
  float eps;
};

constexpr int kTailThreads = 256;

__global__ void __launch_bounds__(kTailThreads)
tail_kernel(const TailArgs a) {
  const int s = blockIdx.x, b = blockIdx.y, S = gridDim.x;
  const int n = s * kTailThreads + threadIdx.x;
  __shared__ float s_ws[32];
  __shared__ float s_warp[kTailThreads / 32];
  __shared__ unsigned s_last;
  if (threadIdx.x < a.k) s_ws[threadIdx.x] = a.topk_w[b * a.k + threadIdx.x];
  __syncthreads();
  float zz = 0.f;
  if (n < a.d) {
    float yr = 0.f;
    const float* yp = a.y_pair + (size_t)b * a.k * a.d + n;
    for (int j = 0; j < a.k; ++j) yr = fmaf(s_ws[j], __ldcg(yp + (size_t)j * a.d), yr);
    const size_t o = (size_t)b * a.d + n;
    const float z = bf16_bits_to_f32(a.residual[o]) + yr + __ldcg(a.y_s + o);
    a.residual[o] = f32_to_bf16_bits(z);
    a.z[o] = z;
    if (a.y_r_dbg) a.y_r_dbg[o] = yr;
    zz = z * z;
  }
  const float ws = warp_sum(zz);
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = ws;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kTailThreads / 32; ++w) t += s_warp[w];
    a.psum[b * S + s] = t;
    __threadfence();
    s_last = (atomicAdd(a.ticket + b, 1u) == (unsigned)(S - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < S; ++i) t += __ldcg(a.psum + b * S + i);
    s_warp[0] = 1.0f / sqrtf(t / (float)a.d + a.eps);
    a.ticket[b] = 0u;
  }
  __syncthreads();
  const float inv = s_warp[0];
  for (int i = threadIdx.x; i < a.d; i += kTailThreads) {
    const size_t o = (size_t)b * a.d + i;
    const float v = __ldcg(a.z + o) * inv * bf16_bits_to_f32(a.gamma[i]);
    a.out[o] = f32_to_bf16_bits(v);
    if (a.out_dbg) a.out_dbg[o] = v;
  }
}

// L2 prefetch of upcoming weights ("What the fused path changes": a small
// kernel walks a table of upcoming weight ranges and pulls them into L2 on a
// third stream).  One prefetch.global.L2::evict_last per 256-byte segment.
struct PrefetchArgs {
  const char* ptr[4];
  size_t bytes[4];
  int n;
};

__global__ void __launch_bounds__(256)
l2_prefetch_kernel(const PrefetchArgs a) {
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (int r = 0; r < a.n; ++r) {
    if (a.bytes[r] == 0) continue;
    const size_t segs = (a.bytes[r] + 255) / 256;
    for (size_t i = tid; i < segs; i += stride) {
      const size_t off = i * 256 < a.bytes[r] ? i * 256 : a.bytes[r] - 1;   // stay inside
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(a.ptr[r] + off));
    }
  }
}

}  // namespace moe
