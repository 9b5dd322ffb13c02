// Router GEMV + sigmoid/bias top-k + routing tables, one kernel.
//
// Structure after "Kimi K3 on GB300: 13 kernels a layer...", section "What
// the fused path changes" (the fused MoE front: router scores, then the
// selection that the routed-expert kernel consumes).  On one GPU the pages'
// TP-sharded router and its NVLink exchange become a grid-wide reduction:
// every CTA writes its experts' logits, and the last CTA to finish (one atomic
// ticket, no spinning) runs top-k and builds the routing tables.
#pragma once

#include "common.cuh"

namespace moe {

struct RouterArgs {
  const uint16_t* x;      // bf16 [B][d]
  const uint16_t* wr;     // bf16 [E][d]
  const float* bias;      // [E]
  int B, d, E, k;
  float routed_scale;
  float* logits;          // workspace [B][E]
  unsigned* done;         // workspace ticket, 0 at rest
  int* x_shift;           // workspace [B]: f16 scaling shift of each x row
  int32_t* topk_idx;      // [B][k]
  float* topk_w;          // [B][k]
  int* n_active;          // number of distinct selected experts
  int* active_expert;     // [n_active] ascending expert ids
  int* active_off;        // [n_active + 1] offsets into pair_list
  int* pair_list;         // [B*k] pair ids p = b*k + j grouped by expert, rows ascending
  unsigned* h_amax;       // [B*k] reset to 0 (max |h| bits per pair, filled by FC1)
  int* work;              // [4] dynamic work counters of the expert kernels, reset to 0
};

constexpr int kRouterWarps = 8;          // 4 experts x 2 K-halves per CTA
constexpr int kRouterExpertsPerCta = 4;
constexpr int kRouterUnroll = 7;         // 16-byte loads in flight per lane

// Logit partials for RB rows of x over one K-half of one expert row.
template <int RB>
__device__ __forceinline__ void router_dot(const RouterArgs& a, int e, int k0, int k1, int b0,
                                           int lane, float (&acc)[RB], float (&amax)[RB],
                                           bool track_amax) {
#pragma unroll
  for (int r = 0; r < RB; ++r) { acc[r] = 0.f; amax[r] = 0.f; }
  const uint16_t* wrow = a.wr + (size_t)e * a.d;
  for (int c0 = k0 + lane * 8; c0 < k1; c0 += 256 * kRouterUnroll) {
    uint4 wv[kRouterUnroll];
#pragma unroll
    for (int u = 0; u < kRouterUnroll; ++u) {
      const int c = c0 + u * 256;
      wv[u] = c < k1 ? ld_stream_u128(wrow + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kRouterUnroll; ++u) {
      const int c = c0 + u * 256;
      if (c < k1) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          if (b0 + r < a.B) {
            const uint4 xv = *reinterpret_cast<const uint4*>(a.x + (size_t)(b0 + r) * a.d + c);
            float s = acc[r];
            s = fma2_bf16(wv[u].x, xv.x, s);
            s = fma2_bf16(wv[u].y, xv.y, s);
            s = fma2_bf16(wv[u].z, xv.z, s);
            s = fma2_bf16(wv[u].w, xv.w, s);
            acc[r] = s;
            if (track_amax) {
              const uint32_t m0 = max(xv.x & 0x7FFFu, xv.x >> 16 & 0x7FFFu);
              const uint32_t m1 = max(xv.y & 0x7FFFu, xv.y >> 16 & 0x7FFFu);
              const uint32_t m2 = max(xv.z & 0x7FFFu, xv.z >> 16 & 0x7FFFu);
              const uint32_t m3 = max(xv.w & 0x7FFFu, xv.w >> 16 & 0x7FFFu);
              amax[r] = fmaxf(amax[r], bf16_bits_to_f32(max(max(m0, m1), max(m2, m3))));
            }
          }
        }
      }
    }
  }
}

// Top-k of one row by a single warp.  Lane l owns experts l, l+32, ...
// Selection compares fp32 (score + bias); ties go to the lower expert id.
__device__ __forceinline__ void router_topk_row(const RouterArgs& a, int b, int lane,
                                                int32_t* s_idx) {
  constexpr int kMaxPerLane = 32;  // E <= 1024
  float key[kMaxPerLane], sc[kMaxPerLane];
#pragma unroll
  for (int m = 0; m < kMaxPerLane; ++m) {
    const int e = m * 32 + lane;
    if (e < a.E) {
      const float l = __ldcg(a.logits + (size_t)b * a.E + e);
      const float s = 1.0f / (1.0f + expf(-l));
      sc[m] = s;
      key[m] = s + __ldg(a.bias + e);
    } else {
      sc[m] = 0.f;
      key[m] = -INFINITY;
    }
  }
  uint32_t taken = 0;
  float ssum = 0.f;
  float sel_s = 0.f;  // score of the j-th pick, kept by lane j
  int sel_e = 0;
  for (int j = 0; j < a.k; ++j) {
    float bv = -INFINITY, bs = 0.f;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int m = 0; m < kMaxPerLane; ++m) {
      const int e = m * 32 + lane;
      if (e < a.E && !(taken >> m & 1u) && key[m] > bv) { bv = key[m]; be = e; bs = sc[m]; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      const float os = __shfl_xor_sync(0xffffffffu, bs, o);
      if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; bs = os; }
    }
    if (be >= a.E) be = 0;   // only reachable with NaN scores; keeps every index in range
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) { sel_e = be; sel_s = bs; }
    ssum += bs;  // identical on all lanes: picks are summed in order j = 0..k-1
  }
  if (lane < a.k) {
    s_idx[b * a.k + lane] = sel_e;
    a.topk_idx[b * a.k + lane] = sel_e;
    a.topk_w[b * a.k + lane] = a.routed_scale * sel_s / ssum;
  }
}

template <int RB>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_topk_kernel(const RouterArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterExpertsPerCta + (warp >> 1);
  const int half = warp & 1;
  const int kh = a.d / 2;
  const int k0 = half * kh, k1 = k0 + kh;
  __shared__ float s_part[kRouterWarps][8];
  __shared__ float s_amax[2][8];
  __shared__ unsigned s_last;
  const bool track = blockIdx.x == 0 && warp < 2;

  for (int b0 = 0; b0 < a.B; b0 += RB) {
    float acc[RB], amax[RB];
    if (e < a.E) {
      router_dot<RB>(a, e, k0, k1, b0, lane, acc, amax, track);
    } else {
#pragma unroll
      for (int r = 0; r < RB; ++r) { acc[r] = 0.f; amax[r] = 0.f; }
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const float s = warp_sum(acc[r]);
      if (lane == 0) s_part[warp][r] = s;
      if (track) {
        const float m = warp_max(amax[r]);
        if (lane == 0) s_amax[warp][r] = m;
      }
    }
    __syncthreads();
    if (half == 0 && lane < RB && e < a.E && b0 + lane < a.B) {
      a.logits[(size_t)(b0 + lane) * a.E + e] = s_part[warp][lane] + s_part[warp + 1][lane];
    }
    if (track && warp == 0 && lane < RB && b0 + lane < a.B) {
      a.x_shift[b0 + lane] = f16_shift_for_amax(fmaxf(s_amax[0][lane], s_amax[1][lane]));
    }
    __syncthreads();
  }

  // ---- grid-wide completion: the last CTA to arrive runs the selection ----
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.done, 1u) == gridDim.x - 1) ? 1u : 0u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  __shared__ int32_t s_idx[64 * 32];              // B*k <= 2048
  __shared__ unsigned long long s_mask[1024];     // rows selecting each expert (B <= 64)
  __shared__ int s_cnt_scan[kRouterWarps * 32];
  __shared__ int s_act_scan[kRouterWarps * 32];

  for (int b = warp; b < a.B; b += kRouterWarps) router_topk_row(a, b, lane, s_idx);
  for (int i = threadIdx.x; i < a.E; i += blockDim.x) s_mask[i] = 0ull;
  __syncthreads();
  const int P = a.B * a.k;
  for (int p = threadIdx.x; p < P; p += blockDim.x)
    atomicOr(&s_mask[s_idx[p]], 1ull << (p / a.k));
  __syncthreads();

  // exclusive scans over experts (ascending ids) of: pair counts, active flags
  const int per = (a.E + blockDim.x - 1) / blockDim.x;
  const int e_lo = threadIdx.x * per;
  int my_cnt = 0, my_act = 0;
  for (int i = 0; i < per; ++i) {
    const int ee = e_lo + i;
    if (ee < a.E) {
      const int c = __popcll(s_mask[ee]);
      my_cnt += c;
      my_act += c > 0;
    }
  }
  // block-wide exclusive scan of (my_cnt, my_act): warp shuffles, then warp totals
  int inc_c = my_cnt, inc_a = my_act;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int tc = __shfl_up_sync(0xffffffffu, inc_c, o);
    const int ta = __shfl_up_sync(0xffffffffu, inc_a, o);
    if (lane >= o) { inc_c += tc; inc_a += ta; }
  }
  if (lane == 31) { s_cnt_scan[warp] = inc_c; s_act_scan[warp] = inc_a; }
  __syncthreads();
  int base_c = 0, base_a = 0;
  for (int w = 0; w < warp; ++w) { base_c += s_cnt_scan[w]; base_a += s_act_scan[w]; }
  if (threadIdx.x == blockDim.x - 1) {
    *a.n_active = base_a + inc_a;
    a.active_off[base_a + inc_a] = base_c + inc_c;
  }
  const int excl_c = base_c + inc_c - my_cnt, excl_a = base_a + inc_a - my_act;
  __syncthreads();
  s_cnt_scan[threadIdx.x] = excl_c;
  s_act_scan[threadIdx.x] = excl_a;
  __syncthreads();
  {
    int off = s_cnt_scan[threadIdx.x], slot = s_act_scan[threadIdx.x];
    for (int i = 0; i < per; ++i) {
      const int ee = e_lo + i;
      if (ee < a.E) {
        const unsigned long long m = s_mask[ee];
        if (m) {
          a.active_expert[slot] = ee;
          a.active_off[slot] = off;
          // pairs of this expert, rows ascending
          unsigned long long mm = m;
          int pos = off;
          while (mm) {
            const int b = __ffsll((long long)mm) - 1;
            mm &= mm - 1;
            int j = 0;
            for (; j < a.k; ++j)
              if (s_idx[b * a.k + j] == ee) break;
            a.pair_list[pos++] = b * a.k + j;
          }
          off += __popcll(m);
          ++slot;
        }
      }
    }
  }
  for (int p = threadIdx.x; p < P; p += blockDim.x) a.h_amax[p] = 0u;
  if (threadIdx.x < 4) a.work[threadIdx.x] = 0;
  if (threadIdx.x == 0) *a.done = 0u;
}

}  // namespace moe
