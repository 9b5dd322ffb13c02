// MoE tail: weighted combine of the routed experts + shared expert + residual,
// then RMSNorm, in one kernel ("Kimi K3 on GB300: 13 kernels a layer...",
// section "What the fused path changes": the tail folds the down-projection
// reduction and the next norm together; at one GPU the reduction is local).
//
// Each row is handled by one thread-block cluster of kTailCluster CTAs; CTA c
// owns d / kTailCluster elements, four per thread.  A thread forms
//   z = residual + sum_j w[b][j] * y_pair[b*k + j] + y_s
// for its elements (all k partial loads issued before use), the CTAs exchange
// their sums of squares through distributed shared memory, and every CTA
// normalises its own elements: out = bf16(z / sqrt(mean z^2 + eps) * gamma).
// The partial sums are added in CTA-rank order, so the result is deterministic.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace moe {

struct TailArgs {
  const float* y_pair;     // [B*k][d]
  const float* topk_w;     // [B][k]
  const float* y_s;        // [B][d]
  const uint16_t* gamma;   // bf16 [d]
  uint16_t* residual;      // bf16 [B][d] in / out
  uint16_t* out;           // bf16 [B][d]
  float* y_r_dbg;          // optional export [B][d]
  float* z_dbg;            // optional export of z before bf16 rounding [B][d]
  float* out_dbg;          // optional export of out before bf16 rounding [B][d]
  int B, d, k;
  float eps;
  unsigned long long* trace;  // optional kernel trace, or null
  // zeroed for the next forward once every earlier kernel of this one has
  // finished: the per-pair max |h| that FC1's epilogues raise
  unsigned* h_amax;           // [B*k]
  // optional L2 prefetch of static weights of the next layer (no dependency:
  // issued before the wait for the predecessor), or null / 0
  const char* pref;
  size_t pref_bytes;
};

constexpr int kTailCluster = 8;
constexpr int kTailBatch = 16;   // y_pair loads in flight per thread

__global__ void __cluster_dims__(kTailCluster, 1, 1) __launch_bounds__(256)
tail_kernel(const TailArgs a) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int c = (int)cluster.block_rank(), b = blockIdx.y;
  const int per_cta = a.d / kTailCluster;
  const int n = c * per_cta + (int)threadIdx.x * 4;
  const bool ok = (int)threadIdx.x * 4 < per_cta;
  __shared__ float s_warp[8];
  __shared__ float s_part[kTailCluster];
  __shared__ float s_w[32];   // the row's combine weights (k <= 32)
  trace_begin(a.trace, 4);
  // first cluster phase: every CTA of the cluster has started (required before
  // any remote shared-memory store); arrive now, wait just before the stores
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  // gamma is a static weight: it may be read before the predecessor finishes
  uint2 g = make_uint2(0, 0);
  if (ok) g = *reinterpret_cast<const uint2*>(a.gamma + n);
  if (a.pref_bytes) {
    // one prefetch.global.L2::evict_last per 256-byte segment, spread over
    // every thread of the grid
    const size_t segs = (a.pref_bytes + 255) / 256;
    const size_t nt = (size_t)gridDim.x * gridDim.y * blockDim.x;
    const size_t t0 = ((size_t)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
    for (size_t i = t0; i < segs; i += nt) {
      const size_t off = i * 256 < a.pref_bytes ? i * 256 : a.pref_bytes - 1;   // stay inside
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(a.pref + off));
    }
  }
  pdl_launch_dependents();
  pdl_wait_prerequisites();
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int i = threadIdx.x; i < a.B * a.k; i += blockDim.x) a.h_amax[i] = 0u;
  }
  float z[4] = {0.f, 0.f, 0.f, 0.f};
  float yr[4] = {0.f, 0.f, 0.f, 0.f};
  // the row's k combine weights, read once per CTA (not once per thread)
  for (int i = threadIdx.x; i < a.k; i += blockDim.x) s_w[i] = __ldcg(a.topk_w + b * a.k + i);
  const size_t o = (size_t)b * a.d + n;
  const float* yp = a.y_pair + (size_t)b * a.k * a.d + n;
  // every load of this thread is issued before the first use: the first
  // batch of pair rows goes out before the barrier that publishes s_w
  float4 ys = make_float4(0.f, 0.f, 0.f, 0.f);
  uint2 rb = make_uint2(0u, 0u);
  float4 v[kTailBatch];
#pragma unroll
  for (int j = 0; j < kTailBatch; ++j) {
    v[j] = ok && j < a.k ? __ldcg(reinterpret_cast<const float4*>(yp + (size_t)j * a.d))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (ok) {
    ys = __ldcg(reinterpret_cast<const float4*>(a.y_s + o));
    rb = __ldcg(reinterpret_cast<const uint2*>(a.residual + o));
  }
  __syncthreads();
  if (ok) {
    for (int j0 = 0; j0 < a.k; j0 += kTailBatch) {
      if (j0 > 0) {
#pragma unroll
        for (int j = 0; j < kTailBatch; ++j)
          v[j] = j0 + j < a.k
                     ? __ldcg(reinterpret_cast<const float4*>(yp + (size_t)(j0 + j) * a.d))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kTailBatch; ++j) {
        const float w = j0 + j < a.k ? s_w[j0 + j] : 0.f;
        yr[0] = fmaf(w, v[j].x, yr[0]);
        yr[1] = fmaf(w, v[j].y, yr[1]);
        yr[2] = fmaf(w, v[j].z, yr[2]);
        yr[3] = fmaf(w, v[j].w, yr[3]);
      }
    }
    z[0] = bf16_bits_to_f32(rb.x & 0xFFFFu) + yr[0] + ys.x;
    z[1] = bf16_bits_to_f32(rb.x >> 16) + yr[1] + ys.y;
    z[2] = bf16_bits_to_f32(rb.y & 0xFFFFu) + yr[2] + ys.z;
    z[3] = bf16_bits_to_f32(rb.y >> 16) + yr[3] + ys.w;
    uint2 ro;
    ro.x = (uint32_t)f32_to_bf16_bits(z[0]) | ((uint32_t)f32_to_bf16_bits(z[1]) << 16);
    ro.y = (uint32_t)f32_to_bf16_bits(z[2]) | ((uint32_t)f32_to_bf16_bits(z[3]) << 16);
    *reinterpret_cast<uint2*>(a.residual + o) = ro;
    if (a.y_r_dbg) *reinterpret_cast<float4*>(a.y_r_dbg + o) = make_float4(yr[0], yr[1], yr[2], yr[3]);
    if (a.z_dbg) *reinterpret_cast<float4*>(a.z_dbg + o) = make_float4(z[0], z[1], z[2], z[3]);
  }
  const float ss = warp_sum(z[0] * z[0] + z[1] * z[1] + z[2] * z[2] + z[3] * z[3]);
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = ss;
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (threadIdx.x < kTailCluster) {
    // every CTA pushes its partial sum into slot c of every peer's s_part
    float t = 0.f;
    for (int w = 0; w < (int)((blockDim.x + 31) >> 5); ++w) t += s_warp[w];
    *cluster.map_shared_rank(&s_part[c], (int)threadIdx.x) = t;
  }
  cluster.sync();   // all pushes have landed; nothing remote is touched after this
  float total = 0.f;
  for (int r = 0; r < kTailCluster; ++r) total += s_part[r];
  const float inv = 1.0f / sqrtf(total / (float)a.d + a.eps);
  if (ok) {
    const size_t o = (size_t)b * a.d + n;
    float v[4];
    v[0] = z[0] * inv * bf16_bits_to_f32(g.x & 0xFFFFu);
    v[1] = z[1] * inv * bf16_bits_to_f32(g.x >> 16);
    v[2] = z[2] * inv * bf16_bits_to_f32(g.y & 0xFFFFu);
    v[3] = z[3] * inv * bf16_bits_to_f32(g.y >> 16);
    uint2 oo;
    oo.x = (uint32_t)f32_to_bf16_bits(v[0]) | ((uint32_t)f32_to_bf16_bits(v[1]) << 16);
    oo.y = (uint32_t)f32_to_bf16_bits(v[2]) | ((uint32_t)f32_to_bf16_bits(v[3]) << 16);
    *reinterpret_cast<uint2*>(a.out + o) = oo;
    if (a.out_dbg) *reinterpret_cast<float4*>(a.out_dbg + o) = make_float4(v[0], v[1], v[2], v[3]);
  }
  trace_end(a.trace, 4);
}

}  // namespace moe
