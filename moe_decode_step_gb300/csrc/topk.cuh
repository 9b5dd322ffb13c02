// Router selection: sigmoid scores, biased top-k per row, combine weights, and
// the routing tables the expert kernels consume.
//
// One CTA per row, one thread per expert (E <= 1024).  Each key is the
// order-preserving unsigned image of the fp32 (score + bias) in the high word
// and the complemented expert id in the low word, so keys are distinct and a
// larger key means a better expert, ties going to the lower id.  Every warp
// sorts its 32 keys (bitonic network over shuffles); then the sorted lists
// meet in a tournament: in each round a warp merges two lists (the elementwise
// maximum of one list and the other reversed is a bitonic sequence holding the
// 32 largest keys of both, which five shuffle stages sort), halving the
// number of lists until one holds the row's 32 best keys in order.  Selection
// compares fp32 (score + bias); the combine weights use the unbiased scores,
// normalised to routed_scale.  The last CTA to finish (atomic ticket, no
// waiting) groups the (row, slot) pairs by expert.  ("Kimi K3 on GB300: 13
// kernels a layer...", section "What one decode step of Kimi K3 does": 16 of
// 896 experts per token.)
#pragma once

#include "common.cuh"

namespace moe {

struct TopkArgs {
  const float* logits;    // [B][E]
  const float* bias;      // [E]
  int B, d, E, k;
  float routed_scale;
  int32_t* topk_idx;      // [B][k], descending by biased score
  float* topk_w;          // [B][k]
  unsigned* done;         // ticket, 0 at rest
  int* n_active;          // routing tables (see RoutedArgs)
  int* active_expert;
  int* active_off;
  int* pair_list;
  unsigned* h_amax;       // [B*k] reset to 0
  unsigned long long* trace;  // optional kernel trace, or null
  unsigned* reset_counts; // if non-null: two done counters of the expert kernels, zeroed
                          // (the router before this kernel ran alone: nothing of the
                          // previous forward still reads them)
};

constexpr int kTopkThreads = 1024;

__device__ __forceinline__ uint32_t float_order_bits(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive block scan of one int per thread (1024 threads); returns the
// exclusive prefix, writes the total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? s_warp[lane] : 0;
    int winc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += t;
    }
    if (lane < nw) s_warp[lane] = winc - w;
    if (lane == nw - 1) s_warp[32] = winc;
  }
  __syncthreads();
  const int r = s_warp[warp] + inc - v;
  *total = s_warp[32];
  __syncthreads();
  return r;
}

// Descending bitonic sort of a bitonic sequence of 32 keys held one per lane.
__device__ __forceinline__ uint64_t warp_bitonic_merge_desc(uint64_t key, int lane) {
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, key, stride);
    const bool lower = (lane & stride) == 0;
    key = lower ? (o > key ? o : key) : (o < key ? o : key);
  }
  return key;
}

// Descending bitonic sort of 32 keys held one per lane.
__device__ __forceinline__ uint64_t warp_bitonic_sort_desc(uint64_t key, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t ok = __shfl_xor_sync(0xffffffffu, key, stride);
      const bool desc = (lane & size) == 0 || size == 32;
      const bool lower = (lane & stride) == 0;
      const bool take = (lower == desc) ? (ok > key) : (ok < key);
      if (take) key = ok;
    }
  }
  return key;
}

// The router's score of one logit, sigma(l), in fp32.
__device__ __forceinline__ float topk_score(float logit) { return 1.0f / (1.0f + expf(-logit)); }

// Selection key of expert e: the order-preserving image of fp32 (score + bias)
// above the complemented id, so a larger key is a better expert and equal
// biased scores go to the lower id.
__device__ __forceinline__ uint64_t topk_key(float score, float bias, int e) {
  return ((uint64_t)float_order_bits(score + bias) << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e);
}

// Expert id of a key.
__device__ __forceinline__ int topk_key_expert(uint64_t key) {
  return (int)(0xFFFFFFFFu - (uint32_t)key);
}

static __global__ void __launch_bounds__(kTopkThreads, 1) topk_kernel(const TopkArgs a) {
  const int b = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  __shared__ int s_warp[33];
  __shared__ float s_score[32];
  __shared__ float s_sc[kTopkThreads];             // sigmoid score of expert t
  __shared__ int32_t s_idx[64 * 32];
  __shared__ unsigned s_last;
  // tournament lists (ping-pong), later reused as the expert masks
  __shared__ __align__(16) uint64_t s_list[2][32][32];
  trace_begin(a.trace, 1);
  // the bias is a static weight: it may be read before the predecessor finishes
  const bool valid = t < a.E;
  const float bias = valid ? __ldg(a.bias + t) : 0.f;
  pdl_launch_dependents();
  pdl_wait_prerequisites();
  if (a.reset_counts && b == 0 && t < 2) a.reset_counts[t] = 0u;

  // ---- scores and keys ----
  uint64_t key = 0ull;
  if (valid) {
    const float score = topk_score(__ldcg(a.logits + (size_t)b * a.E + t));
    s_sc[t] = score;
    key = topk_key(score, bias, t);
  }
  // ---- per-warp bitonic sort, descending ----
  key = warp_bitonic_sort_desc(key, lane);
  // ---- tournament of the sorted warp lists ----
  int n = (a.E + 31) >> 5;   // lists holding valid keys
  if (warp < n) s_list[0][warp][lane] = key;
  __syncthreads();
  int src = 0;
  while (n > 1) {
    const int half = n >> 1;
    if (warp < half) {
      const uint64_t x = s_list[src][2 * warp][lane];
      const uint64_t y = s_list[src][2 * warp + 1][31 - lane];
      s_list[src ^ 1][warp][lane] = warp_bitonic_merge_desc(x > y ? x : y, lane);
    } else if (warp == half && (n & 1)) {
      s_list[src ^ 1][warp][lane] = s_list[src][n - 1][lane];
    }
    n = half + (n & 1);
    src ^= 1;
    __syncthreads();
  }
  if (warp == 0) {
    if (lane < a.k) {
      const int e = topk_key_expert(s_list[src][0][lane]);
      a.topk_idx[b * a.k + lane] = e;
      s_idx[b * a.k + lane] = e;
      s_score[lane] = s_sc[e];
    }
    __syncwarp();
    float ssum = 0.f;
    for (int i = 0; i < a.k; ++i) ssum += s_score[i];   // picks summed in rank order
    if (lane < a.k) a.topk_w[b * a.k + lane] = a.routed_scale * s_score[lane] / ssum;
    if (lane < a.k) a.h_amax[b * a.k + lane] = 0u;
    if (gridDim.x == 1 && a.B == 1) {
      // one row: the k experts are distinct, each with one pair; the tables
      // list them by expert id (slot = rank of the id among the k), pair =
      // rank by score.  Nothing else to build.
      const int e = lane < a.k ? s_idx[lane] : 0x7FFFFFFF;
      int slot = 0;
      for (int i = 0; i < a.k; ++i) slot += s_idx[i] < e ? 1 : 0;
      if (lane < a.k) {
        a.active_expert[slot] = e;
        a.active_off[lane] = lane;
        a.pair_list[slot] = lane;
      }
      if (lane == 0) {
        *a.n_active = a.k;
        a.active_off[a.k] = a.k;
      }
    }
  }
  if (gridDim.x == 1 && a.B == 1) {
    trace_end(a.trace, 1);
    return;
  }
  // ---- the last CTA groups pairs by expert ----
  if (gridDim.x > 1) {
    __threadfence();
    __syncthreads();
    if (t == 0) s_last = (atomicAdd(a.done, 1u) == (unsigned)(gridDim.x - 1)) ? 1u : 0u;
    __syncthreads();
    if (!s_last) {
      trace_end(a.trace, 1);
      return;
    }
    __threadfence();
  } else {
    __syncthreads();
  }
  unsigned long long* s_mask = reinterpret_cast<unsigned long long*>(&s_list[0][0][0]);
  const int P = a.B * a.k;
  if (gridDim.x > 1)   // other rows were selected by other CTAs
    for (int p = t; p < P; p += blockDim.x) s_idx[p] = __ldcg(a.topk_idx + p);
  if (valid) s_mask[t] = 0ull;
  __syncthreads();
  for (int p = t; p < P; p += blockDim.x) atomicOr(&s_mask[s_idx[p]], 1ull << (p / a.k));
  __syncthreads();
  const unsigned long long mask = valid ? s_mask[t] : 0ull;
  const int cnt = __popcll(mask);
  int total_pairs, n_act;
  const int off = block_exclusive_scan(cnt, s_warp, &total_pairs);
  const int slot = block_exclusive_scan(cnt > 0 ? 1 : 0, s_warp, &n_act);
  // each expert's first pair position (the scores are no longer needed)
  int* s_off = reinterpret_cast<int*>(s_sc);
  if (valid) s_off[t] = off;
  if (cnt > 0) {
    a.active_expert[slot] = t;
    a.active_off[slot] = off;
  }
  __syncthreads();
  // pair p = row * k + j goes to its expert's list at the rank of its row
  // among the expert's rows (ascending)
  for (int p = t; p < P; p += blockDim.x) {
    const int e = s_idx[p], row = p / a.k;
    const unsigned long long below = (1ull << row) - 1ull;
    a.pair_list[s_off[e] + __popcll(s_mask[e] & below)] = p;
  }
  if (t == 0) {
    *a.n_active = n_act;
    a.active_off[n_act] = total_pairs;
    if (gridDim.x > 1) *a.done = 0u;
  }
  trace_end(a.trace, 1);
}

}  // namespace moe
